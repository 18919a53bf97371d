"""Host logic of bench.py that needs no GPU: the reference arm's sample fitting and the oracle
step on a head subset (CPU only)."""
import pytest

import bench
from workload import make_batch


class _Req:
    def __init__(self, n_rows):
        self.n_rows = n_rows


class _B:
    def __init__(self, hkv, rows):
        self.hkv = hkv
        self.requests = [_Req(r) for r in rows]


@pytest.mark.parametrize("w_fixed,w_attn,budget", [(0.5, 4.0, 10.0), (0.5, 4.0, 0.7), (2.0, 8.0, 0.4),
                                                   (0.1, 0.1, 0.001)])
def test_fit_sample_meets_the_budget_or_its_limits(w_fixed, w_attn, budget):
    b = _B(hkv=8, rows=[1776])
    stride, hdiv = bench._fit_sample(b, [0], 16, w_fixed, w_attn, budget)
    est = (w_fixed + w_attn * 16 / stride) / hdiv
    max_stride = 1776 // 16
    assert stride >= 16 and stride <= max(16, max_stride) and b.hkv % hdiv == 0
    # within budget, or every knob at its limit (at least 16 rows a request, one kv head)
    assert est <= budget or (stride * 2 > max_stride and hdiv == b.hkv)
    if (w_fixed + w_attn) <= budget:
        assert (stride, hdiv) == (16, 1)          # nothing coarsened when the base sample fits


def test_oracle_step_on_a_head_subset_counts_the_same_tokens():
    b = make_batch("tiny")
    prep = bench.oracle_prepare(b)
    ids = list(range(len(b.requests)))
    t1, s1, f1, a1 = bench.oracle_step(b, prep, ids, 1, 1)
    t2, s2, f2, a2 = bench.oracle_step(b, prep, ids, 1, 2)
    assert t1 == t2 == sum(r.n_cached + r.n_query for r in b.requests)
    assert s1 > 0 and s2 > 0 and f2 >= 0 and a2 >= 0
    # the scaled time counts the subset's work twice (the head subset halves the heads)
    assert s2 == pytest.approx(2 * (f2 + a2), rel=1e-9)
