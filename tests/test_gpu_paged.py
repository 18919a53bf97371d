"""GPU parity of the paged calls (pcf_score_paged, pcf_fused_attention_paged): cached key (and
value) tiles copied straight from the pool pages through the block table, the keys rotated in
shared memory to the request's positions before the tensor-core contraction (MiniPIC 2.1), and in
the attention each recomputed token's fresh key and value written over its stale cached copy in
place.  Every case is checked against the fp64 oracle -- importance within 1e-3 relative, the
attention with the oracle's selection within 2e-2 absolute + 1e-2 relative -- like the compacted
calls; the two kinds of call are also compared with each other."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import method
from workload import make_batch, small_custom_batch

from gpu_util import GpuBatch, assert_close_out
from test_gpu_parity import check_batch, gpu_batch

pytestmark = pytest.mark.gpu


def test_paged_tiny_full():
    check_batch(gpu_batch("tiny"), paged=True)


def test_paged_llama8b_layer_full():
    check_batch(gpu_batch("llama8b_layer"), paged=True)


def test_paged_concurrent_reuse_sampled():
    check_batch(gpu_batch("concurrent_reuse"), req_ids=[0, 7, 31], sample_rows=True, paged=True)


@pytest.mark.parametrize("pct", [5, 15, 30])
def test_paged_long_context_sampled(pct):
    # 30 %: about 38 recomputed tokens per 128-key tile, more than the 32 fresh keys staged with a
    # tile, so the rest are read from global memory
    check_batch(gpu_batch("long_context", pct), sample_rows=True, paged=True)


def test_paged_batch70b_sampled():
    check_batch(gpu_batch("batch70b"), req_ids=[0, 63], sample_rows=True, paged=True)


def test_paged_offset_0_and_2048_share_physical_pages():
    b = small_custom_batch([(0, 8, 0, 20)], n_query=16, hq=8, hkv=2, d=128, theta=5e5,
                           extra_requests=[([(0, 8, 2048, 20)], 16, 2048 + 128)])
    check_batch(GpuBatch(b), paged=True)


def test_paged_full_recompute_equals_full_prefill():
    # every cached key is replaced by its fresh row: 128 per tile, far beyond the staged block
    b = small_custom_batch([(0, 4, 0, 64), (4, 3, 64, 48)], n_query=9, hq=8, hkv=2, d=128, theta=5e5)
    gb = GpuBatch(b)
    r = b.requests[0]
    sel = np.arange(r.n_cached)
    excl, row_pos = gb.selection_inputs([sel])
    out = gb.attention(excl, row_pos, paged=True)
    exp = method.full_prefill(b.q_fresh.double().numpy(), b.k_fresh.double().numpy(),
                              b.v_fresh.double().numpy(), row_pos.astype(np.int64), b.theta)
    assert_close_out(out, exp, "100% recompute, paged")


@pytest.mark.parametrize("case", [
    dict(spans=[(0, 1, 0, 0)], n_query=1),
    dict(spans=[(0, 2, 5, 32)], n_query=3),
    dict(spans=[(0, 3, 0, 1), (3, 5, 48, 7), (8, 1, 200, 16)], n_query=7),
    dict(spans=[], n_query=5),
    dict(spans=[(0, 9, 0, 30)], n_query=0),
])
@pytest.mark.parametrize("shape", [dict(hq=4, hkv=4, d=64), dict(hq=16, hkv=2, d=128)])
def test_paged_edge_cases(case, shape):
    b = small_custom_batch(case["spans"], case["n_query"], n_phys_pages=12, theta=1e4, **shape)
    check_batch(GpuBatch(b), paged=True)


def test_paged_mixed_requests_in_one_batch():
    b = small_custom_batch([(0, 3, 7, 5)], n_query=2, hq=8, hkv=2, d=128, theta=5e5, n_phys_pages=40,
                           extra_requests=[([(3, 17, 100, 40), (20, 9, 2000, 3)], 33, 3000),
                                           ([], 4, 10),
                                           ([(0, 3, 9000, 48), (29, 11, 9100, 100)], 130, 9400)])
    check_batch(GpuBatch(b), paged=True)


@pytest.mark.parametrize("name", ["llama8b_layer", "long_context"])
def test_paged_and_compacted_agree_and_paged_is_deterministic(name):
    gb = gpu_batch(name)
    gb.score()
    gb.topk()
    a = gb.attention().copy()
    p1 = gb.attention(paged=True).copy()
    p2 = gb.attention(paged=True).copy()
    assert np.array_equal(p1.view(np.uint32), p2.view(np.uint32))
    # the two calls round differently (rotation in fp32 from a stepped angle vs a table row), so
    # they agree to the bf16 output precision, not bit for bit
    err = np.abs(p1 - a)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(a)), f"max diff {err.max():.3e}"


@pytest.mark.parametrize("name", ["llama8b_layer", "long_context"])
def test_paged_and_compacted_scoring_agree_and_paged_is_deterministic(name):
    gb = gpu_batch(name)
    a = gb.score().copy()
    p1 = gb.score(paged=True).copy()
    p2 = gb.score(paged=True).copy()
    assert np.array_equal(p1.view(np.uint32), p2.view(np.uint32))
    err = np.abs(p1 - a)
    assert np.all(err <= 2e-3 * np.abs(a) + 1e-7), f"max rel diff {(err / np.maximum(a, 1e-30)).max():.3e}"


def test_paged_step_through_the_public_api_matches_the_compacted_one():
    """CacheFusion(paged=True): scoring, top-k and attention with no copy of the cached keys or
    values; the selection equals the compacted pipeline's wherever the two importances do not tie
    within rounding, and the output matches the oracle given that selection."""
    import position_independent_kv_critical_gb300 as pcf
    b = make_batch("llama8b_layer")
    gb = GpuBatch(b)
    cfp = pcf.CacheFusion(gb.L, gb.rope, device="cuda", paged=True)
    cfp.step(gb.q_query, gb.k_pool, gb.v_pool, gb.q_fresh, gb.k_fresh, gb.v_fresh)
    pcf.check_device_error()
    sel = cfp.sel_idx[: gb.L.total_sel].cpu().numpy().astype(np.int64)
    exp, _ = gb.oracle_attention(0, sel)
    got = cfp.out[: gb.L.total_rows].float().cpu().numpy()
    assert_close_out(got, exp, "paged step")
