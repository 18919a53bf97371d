"""fp64 CPU oracle for query-centric cache fusion over a position-free KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this package:
it is used by ``tests/``, by ``__graft_entry__.smoke()`` (to check one small GPU call) and by the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It shares no code with the CUDA
path (no kernels, headers, helpers or constants); the two meet only in the seeded inputs of
``workload/``.

What it computes, and from which passage:

* ``rope``   rotary position embedding R_p applied to an unrotated vector, used to rotate cached
  keys at their per-request logical position pi(j) and queries at theirs
  (MiniPIC: Position-Independent Caching ..., section 2.1 "Position-free KV", score equation).
* ``method.score_request``  critical-layer attention of the query tokens over the request's cached
  keys only, summed over heads and query tokens into one importance value per cached token
  (QCFuse: Query-Centric Cache Fusion ..., section 2B "Critical-layer attention profiling";
  second summary, Phase 3 "only the key cache of one critical layer").
* ``method.score_layers_request``  the same importance taken at every layer and summed over the
  layers (the all-layer comparison point of QCFuse section 4 "Resultados", QCAll).
* ``method.select_topk_request``  the tokens with the highest importance, chosen per span, ties to
  the lower index (QCFuse section 2B "Top-N tokens"; per-span selection is the workload's reading).
* ``method.fused_attention_request``  causal attention of the recomputed rows and the query rows
  over the cached keys minus the recomputed tokens plus the fresh rows, every key rotated at its
  logical position (QCFuse section 2C / Phase 4 "discrete recomputation", causal constraints of
  the sparse-attention kernel; MiniPIC section 2.1 score equation).
* ``method.full_prefill``  plain causal prefill over given rows, written separately as the
  100 %-recompute reference.

Parity pins live in ``tests/test_oracle_pins.py``.  Every function above has at least one pin that
does not go through the oracle itself.
"""
from . import rope, method  # noqa: F401
