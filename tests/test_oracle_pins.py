"""Pins of the fp64 oracle against facts the pages and the mathematics fix (CPU only).

Each check goes through something other than the oracle itself: a closed form, an invariant,
a library routine (scipy expm, torch scaled_dot_product_attention) or brute force in plain Python.
Chosen so that a plausible mistake (wrong rotation sign or pairing, a dropped 1/sqrt(d), softmax
over the wrong axis, a transposed operand, the wrong GQA head map, inverted causal mask, a bad
tie rule) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import method, rope
from workload import CONFIGS, make_layout, small_custom_batch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------- independent rotation forms ----------

def _freqs(d, theta):
    return np.array([theta ** (-2.0 * i / d) for i in range(d // 2)])


def rot_expm(x, p, theta):
    """R_p x via the matrix exponential of the rotation generator (scipy)."""
    d = x.shape[-1]
    h = d // 2
    f = _freqs(d, theta)
    G = np.zeros((d, d))
    for i in range(h):
        G[i, i + h] = -f[i]
        G[i + h, i] = f[i]
    return scipy.linalg.expm(p * G) @ x


def rot_complex(x, pos, theta):
    """R_p x as complex multiplication z_i * exp(i p f_i), z_i = x_i + 1j x_{i+d/2}."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    f = _freqs(d, theta)
    pos = np.asarray(pos, dtype=np.float64).reshape((-1,) + (1,) * (x.ndim - 1))
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * f)
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("d,theta", [(8, 1e4), (16, 5e5), (64, 1e4)])
@pytest.mark.parametrize("p", [0, 1, 7, 513, 2048, 4095])
def test_rotate_matches_matrix_exponential(d, theta, p):
    x = np.random.default_rng(d + p).standard_normal(d)
    got = rope.rotate(x[None], np.array([p]), theta)[0]
    np.testing.assert_allclose(got, rot_expm(x, p, theta), rtol=0, atol=1e-9)


def test_rotate_matches_complex_form_large_positions():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 3, 128))
    pos = rng.integers(0, 65536, size=50)
    np.testing.assert_allclose(rope.rotate(x, pos, 5e5), rot_complex(x, pos, 5e5), atol=1e-12)


def test_rotate_d2_closed_form():
    # d = 2: frequency theta^0 = 1, so R_p = [[cos p, -sin p], [sin p, cos p]]
    for p in [0, 1, 3, 100]:
        e0 = rope.rotate(np.array([[1.0, 0.0]]), np.array([p]), 1e4)[0]
        e1 = rope.rotate(np.array([[0.0, 1.0]]), np.array([p]), 1e4)[0]
        np.testing.assert_allclose(e0, [math.cos(p), math.sin(p)], atol=1e-15)
        np.testing.assert_allclose(e1, [-math.sin(p), math.cos(p)], atol=1e-15)


def test_rotation_norm_and_group_property():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((20, 128))
    a = rng.integers(0, 30000, 20)
    b = rng.integers(0, 30000, 20)
    ra = rope.rotate(x, a, 5e5)
    np.testing.assert_allclose(np.linalg.norm(ra, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(rope.rotate(ra, b, 5e5), rope.rotate(x, a + b, 5e5), atol=1e-9)


def test_on_the_fly_rotation_equals_rerotating_cache_hits():
    """MiniPIC 2.1: rotating the unrotated key at pi(j) in the kernel is algebraically the same as
    re-rotating a cache hit that was stored rotated at offset c by (pi(j) - c)."""
    rng = np.random.default_rng(3)
    k = rng.standard_normal((32, 2, 64))
    c = np.arange(32)                      # stored at offset 0
    pi = 2048 + np.arange(32)              # reused at offset 2048
    stored = rot_complex(k, c, 1e4)
    np.testing.assert_allclose(rope.rotate(stored, pi - c, 1e4), rope.rotate(k, pi, 1e4), atol=1e-10)


def test_score_depends_only_on_relative_position_closed_form():
    # d = 2, q = k = e0: (R_t q).(R_pi k)/sqrt(2) = cos(t - pi)/sqrt(2)
    K = np.array([[[1.0, 0.0]]])
    for t, p in [(5, 2), (2, 5), (1000, 999), (7, 7)]:
        qr = rope.rotate(np.array([[[1.0, 0.0]]]), np.array([t]), 1e4)
        kr = rope.rotate(K, np.array([p]), 1e4)
        s = float(qr[0, 0] @ kr[0, 0]) / math.sqrt(2)
        assert abs(s - math.cos(t - p) / math.sqrt(2)) < 1e-13


# ---------- importance ----------

class _Sp:
    def __init__(self, first, n, pos0, k=0):
        self.phys_first_page, self.n_pages, self.pos0, self.k = first, n, pos0, k


def test_importance_two_key_worked_example():
    # d = 2, all positions 0 (R = I); scores 0 and ln 3 -> weights 1/4 and 3/4
    q = np.array([[[math.sqrt(2.0), 0.0]]])
    K = np.array([[[0.0, 0.0]], [[math.log(3.0), 0.0]]])
    imp = method.score_request(q, np.array([0]), K, np.array([0, 0]), 1e4)
    np.testing.assert_allclose(imp, [0.25, 0.75], atol=1e-15)


def test_importance_sums_to_heads_times_queries_and_uniform_for_zero_query():
    rng = np.random.default_rng(4)
    T, hq, hkv, d, N = 5, 4, 2, 16, 48
    q = rng.standard_normal((T, hq, d))
    K = rng.standard_normal((N, hkv, d))
    kpos = np.arange(N) + 100
    qpos = N + 100 + np.arange(T)
    imp = method.score_request(q, qpos, K, kpos, 1e4)
    assert abs(imp.sum() - hq * T) < 1e-11
    imp0 = method.score_request(np.zeros_like(q), qpos, K, kpos, 1e4)
    np.testing.assert_allclose(imp0, np.full(N, hq * T / N), atol=1e-13)


def test_importance_brute_force_python_loops():
    rng = np.random.default_rng(5)
    T, hq, hkv, d, N = 4, 2, 1, 8, 32
    q = rng.standard_normal((T, hq, d))
    K = rng.standard_normal((N, hkv, d))
    kpos = np.concatenate([3 + np.arange(16), 40 + np.arange(16)])
    qpos = 60 + np.arange(T)
    theta = 1e4
    h2 = d // 2
    f = [theta ** (-2.0 * i / d) for i in range(h2)]

    def rot(v, p):
        out = [0.0] * d
        for i in range(h2):
            c, s = math.cos(p * f[i]), math.sin(p * f[i])
            out[i] = v[i] * c - v[i + h2] * s
            out[i + h2] = v[i + h2] * c + v[i] * s
        return out

    ref = [0.0] * N
    for h in range(hq):
        for t in range(T):
            qr = rot(list(q[t, h]), int(qpos[t]))
            logits = []
            for j in range(N):
                kr = rot(list(K[j, 0]), int(kpos[j]))
                logits.append(sum(a * b for a, b in zip(qr, kr)) / math.sqrt(d))
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            for j in range(N):
                ref[j] += w[j] / z
    np.testing.assert_allclose(method.score_request(q, qpos, K, kpos, theta), ref, atol=1e-12)


# ---------- all-layer importance (QCAll) ----------

def test_layer_importance_sums_to_layers_times_heads_times_queries():
    rng = np.random.default_rng(11)
    L, T, hq, hkv, d, N = 3, 5, 4, 2, 16, 40
    qs = [rng.standard_normal((T, hq, d)) for _ in range(L)]
    Ks = [rng.standard_normal((N, hkv, d)) for _ in range(L)]
    kpos, qpos = 7 + np.arange(N), 50 + np.arange(T)
    per, tot = method.score_layers_request(qs, qpos, Ks, kpos, 1e4)
    assert per.shape == (L, N) and tot.shape == (N,)
    np.testing.assert_allclose(per.sum(axis=1), np.full(L, hq * T), atol=1e-11)
    assert abs(tot.sum() - L * hq * T) < 1e-10


def test_layer_importance_of_identical_layers_is_l_times_one_layer_and_zero_query_is_uniform():
    rng = np.random.default_rng(12)
    T, hq, hkv, d, N = 3, 2, 1, 8, 24
    q = rng.standard_normal((T, hq, d))
    K = rng.standard_normal((N, hkv, d))
    kpos, qpos = np.arange(N), N + np.arange(T)
    one = method.score_request(q, qpos, K, kpos, 1e4)
    per, tot = method.score_layers_request([q] * 4, qpos, [K] * 4, kpos, 1e4)
    np.testing.assert_allclose(tot, 4 * one, rtol=1e-14)
    # a layer whose query is zero spreads its weight evenly: hq*T/N per token (closed form)
    per, tot = method.score_layers_request([q, np.zeros_like(q)], qpos, [K, K], kpos, 1e4)
    np.testing.assert_allclose(per[1], np.full(N, hq * T / N), atol=1e-13)
    np.testing.assert_allclose(tot, one + hq * T / N, rtol=1e-13)


def test_layer_importance_pairs_each_query_with_its_own_layers_keys():
    # two-key worked example per layer (d = 2, positions 0): layer 0 scores 0 and ln 3 (weights
    # 1/4, 3/4), layer 1 the keys swapped (3/4, 1/4); taking layer 0's keys for both layers, or
    # layer 1's query for both, changes the per-layer rows
    q = np.array([[[math.sqrt(2.0), 0.0]]])
    K0 = np.array([[[0.0, 0.0]], [[math.log(3.0), 0.0]]])
    K1 = K0[::-1].copy()
    per, tot = method.score_layers_request([q, q], np.array([0]), [K0, K1], np.array([0, 0]), 1e4)
    np.testing.assert_allclose(per, [[0.25, 0.75], [0.75, 0.25]], atol=1e-15)
    np.testing.assert_allclose(tot, [1.0, 1.0], atol=1e-15)
    q2 = np.array([[[0.0, 0.0]]])     # layer 1's query carries no preference: weights 1/2, 1/2
    per, _ = method.score_layers_request([q, q2], np.array([0]), [K0, K1], np.array([0, 0]), 1e4)
    np.testing.assert_allclose(per, [[0.25, 0.75], [0.5, 0.5]], atol=1e-15)


# ---------- top-k ----------

def _brute_topk(vals, k):
    return sorted(sorted(range(len(vals)), key=lambda i: (-vals[i], i))[:k])


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_planted_ties(seed):
    rng = np.random.default_rng(seed)
    lens = [16, 48, 128, 32]
    vals = rng.integers(0, 12, size=sum(lens)).astype(np.float32) * np.float32(0.125)
    ks = [int(rng.integers(0, L + 1)) for L in lens]
    got = method.select_topk_request(vals, lens, ks)
    exp, off = [], 0
    for L, k in zip(lens, ks):
        exp += [off + i for i in _brute_topk(list(vals[off:off + L]), k)]
        off += L
    assert list(got) == exp


def test_topk_all_equal_takes_first_indices_and_boundary_ties():
    v = np.ones(64, dtype=np.float32)
    assert list(method.select_topk_request(v, [64], [10])) == list(range(10))
    w = np.zeros(32, dtype=np.float32)
    w[[3, 9, 20, 27]] = 5.0       # four equal maxima straddling k = 2
    assert list(method.select_topk_request(w, [32], [2])) == [3, 9]
    assert list(method.select_topk_request(w, [32], [0])) == []
    assert list(method.select_topk_request(w, [32], [32])) == list(range(32))


# ---------- global Top-N (the pages' own reading) ----------

def test_global_topn_worked_example():
    v = np.array([0.1, 0.5, 0.5, 0.2, 0.9], dtype=np.float32)
    assert list(method.select_topn_global_request(v, 2)) == [1, 4]     # 0.9, then the first 0.5
    assert list(method.select_topn_global_request(v, 3)) == [1, 2, 4]
    assert list(method.select_topn_global_request(v, 0)) == []
    assert list(method.select_topn_global_request(v, 5)) == [0, 1, 2, 3, 4]


def test_global_topn_single_span_equals_per_span_selection():
    rng = np.random.default_rng(11)
    vals = rng.integers(0, 9, size=96).astype(np.float32) * np.float32(0.25)
    for k in (0, 1, 17, 50, 96):
        assert list(method.select_topn_global_request(vals, k)) == list(method.select_topk_request(vals, [96], [k]))


@pytest.mark.parametrize("seed", range(5))
def test_global_topn_separates_chosen_from_the_rest(seed):
    """Every chosen value is >= every other value; among values equal to the smallest chosen one,
    the chosen are the lowest indices (checked by counting, not by sorting)."""
    rng = np.random.default_rng(100 + seed)
    vals = rng.integers(0, 6, size=200).astype(np.float32)
    n = int(rng.integers(1, 200))
    sel = method.select_topn_global_request(vals, n)
    assert len(sel) == n and np.all(np.diff(sel) > 0)
    rest = np.setdiff1d(np.arange(200), sel)
    t = vals[sel].min()
    assert len(rest) == 0 or vals[rest].max() <= t
    ties = np.nonzero(vals == t)[0]
    taken = np.intersect1d(ties, sel)
    assert list(taken) == list(ties[:len(taken)])


def test_global_topn_moves_the_budget_across_spans():
    """Two spans of 16 with k = 4 each: per span takes 4 + 4; globally all 8 come from the span
    holding the larger values."""
    v = np.concatenate([np.linspace(1.0, 2.0, 16), np.linspace(0.0, 0.5, 16)]).astype(np.float32)
    per_span = method.select_topk_request(v, [16, 16], [4, 4])
    assert list(per_span) == [12, 13, 14, 15, 28, 29, 30, 31]
    assert list(method.select_topn_global_request(v, 8)) == list(range(8, 16))


# ---------- anchors: key norms and per-span top-m ----------

def test_key_norms_closed_forms():
    K = np.full((3, 8, 128), 0.5)
    np.testing.assert_allclose(method.key_norms(K), 0.5 * math.sqrt(8 * 128), rtol=1e-15)
    E = np.zeros((4, 2, 64))
    E[0, 1, 5] = -3.0
    E[1, 0, 63] = 2.5
    E[3, 1, 0], E[3, 0, 1] = 3.0, 4.0       # a 3-4-5 triangle across two heads
    np.testing.assert_allclose(method.key_norms(E), [3.0, 2.5, 0.0, 5.0], rtol=1e-15)


def test_key_norms_do_not_depend_on_the_position():
    """RoPE is a rotation: the norm of the cached (position-free) key equals that of the key
    rotated to any position, so anchors need no positions."""
    rng = np.random.default_rng(5)
    K = rng.standard_normal((40, 4, 64))
    pos = rng.integers(0, 60000, 40)
    np.testing.assert_allclose(method.key_norms(rope.rotate(K, pos, 5e5)), method.key_norms(K), rtol=1e-12)


def test_anchors_worked_example():
    norms = np.array([1.0, 3.0, 2.0, 3.0, 0.5, 0.5, 4.0, 0.1], dtype=np.float32)
    assert list(method.select_anchors_request(norms, [4, 4], [2, 1])) == [1, 3, 6]


def test_anchor_count_whole_pages():
    assert [method.anchor_count(p, 512) for p in (0, 1, 3, 6, 7, 100)] == [0, 16, 16, 32, 48, 512]
    assert method.anchor_count(5, 1024) == 64


def test_anchor_probe_equals_causal_prefill_over_the_prefixed_sequence():
    """The probe's query rows are the last T rows of a plain causal prefill over [anchors; query]
    at positions 0 .. A+T-1 (the anchors' own query rows do not matter)."""
    rng = np.random.default_rng(21)
    A, T, hq, hkv, d = 32, 6, 4, 2, 16
    Ka, Va = rng.standard_normal((A, hkv, d)), rng.standard_normal((A, hkv, d))
    q, k, v = rng.standard_normal((T, hq, d)), rng.standard_normal((T, hkv, d)), rng.standard_normal((T, hkv, d))
    got = method.anchor_probe_request(q, k, v, Ka, Va, 1e4)
    q_all = np.concatenate([rng.standard_normal((A, hq, d)), q])
    full = method.full_prefill(q_all, np.concatenate([Ka, k]), np.concatenate([Va, v]),
                               np.arange(A + T), 1e4)
    np.testing.assert_allclose(got, full[A:], atol=1e-12)


def test_anchor_probe_without_anchors_is_the_query_alone():
    rng = np.random.default_rng(22)
    T, hq, hkv, d = 5, 2, 1, 8
    q, k, v = rng.standard_normal((T, hq, d)), rng.standard_normal((T, hkv, d)), rng.standard_normal((T, hkv, d))
    z = np.zeros((0, hkv, d))
    got = method.anchor_probe_request(q, k, v, z, z, 1e4)
    # the first query token sees only itself: its output is its own value row
    np.testing.assert_allclose(got[0], np.repeat(v[0], hq // hkv, axis=0), atol=1e-12)
    np.testing.assert_allclose(got, method.full_prefill(q, k, v, np.arange(T), 1e4), atol=1e-12)


def test_k_from_percent_golden_table():
    with open(os.path.join(GOLDEN, "recompute_counts.txt")) as fh:
        rows = [ln.split("#")[0].split() for ln in fh if ln.split("#")[0].strip()]
    assert rows
    for pct, L, k in rows:
        assert method.k_from_percent(int(pct), int(L)) == int(k)


def test_exclusion_masks_bits():
    sel = np.array([0, 5, 15, 16, 31, 47])
    m = method.exclusion_masks(sel, 3)
    for j in range(48):
        assert bool((int(m[j // 16]) >> (j % 16)) & 1) == (j in set(sel.tolist()))


# ---------- row positions and the recompute gather (QCFuse Phase 4: the Top-N indices are
# recomputed at their own positions, then the query follows) ----------

class _Sp:
    def __init__(self, phys_first_page, n_pages, pos0):
        self.phys_first_page, self.n_pages, self.pos0 = phys_first_page, n_pages, pos0


def test_row_positions_worked_example():
    # span A: one page at positions 100..115; span B: two pages at 300..331; query of 3 tokens at
    # 332..334.  Request-local tokens 3 (A), 17 and 30 (B offsets 1 and 14) are recomputed.
    hkv, d = 1, 4
    pool = np.zeros((3, hkv, 16, d))
    _, _, kpos = method.request_cached([_Sp(0, 1, 100), _Sp(1, 2, 300)], pool, pool)
    got = method.row_positions(np.array([3, 17, 30]), kpos, 3, 332)
    assert got.tolist() == [103, 301, 314, 332, 333, 334]


@pytest.mark.parametrize("seed", range(4))
def test_row_positions_ordered_and_query_contiguous(seed):
    rng = np.random.default_rng(seed)
    spans, pos = [], int(rng.integers(0, 4096))
    for i in range(int(rng.integers(1, 6))):
        n = int(rng.integers(1, 5))
        spans.append(_Sp(i * 4, n, pos))
        pos += 16 * n + 16 * int(rng.integers(0, 3))       # spans may leave gaps
    pool = np.zeros((4 * len(spans), 1, 16, 2))
    _, _, kpos = method.request_cached(spans, pool, pool)
    # positions written out span by span, independently of request_cached
    direct = [s.pos0 + t for s in spans for t in range(16 * s.n_pages)]
    n_tok = len(direct)
    sel = np.sort(rng.choice(n_tok, size=int(rng.integers(0, n_tok + 1)), replace=False))
    nq, q0 = int(rng.integers(0, 9)), pos + 5
    got = method.row_positions(sel, kpos, nq, q0)
    assert len(got) == len(sel) + nq
    assert got[: len(sel)].tolist() == [direct[j] for j in sel.tolist()]
    assert np.all(np.diff(got[: len(sel)]) > 0)                 # recomputed rows in position order
    assert got[len(sel):].tolist() == list(range(q0, q0 + nq))  # query rows follow, contiguous
    if len(sel) and nq:
        assert got[len(sel) - 1] < got[len(sel)]


def test_gather_rows_worked_example():
    src = np.arange(15, dtype=np.int64).reshape(5, 3)
    got = method.gather_rows(src, np.array([4, 0, 2]))
    assert got.tolist() == [[12, 13, 14], [0, 1, 2], [6, 7, 8]]
    assert got.dtype == src.dtype
    assert method.gather_rows(src, np.zeros((0,), dtype=np.int64)).shape == (0, 3)


def test_gather_rows_of_an_ascending_selection_keep_the_selection_order():
    # a bf16-exact integer pattern: row j is j*8 + column, so a gathered row names its source
    src = (np.arange(40 * 8, dtype=np.float64).reshape(40, 8))
    sel = np.array([1, 2, 7, 19, 33, 39])
    got = method.gather_rows(src, sel)
    assert [int(r[0]) // 8 for r in got] == sel.tolist()
    assert all(np.array_equal(r, np.arange(8) + 8 * j) for r, j in zip(got, sel))


# ---------- attention ----------

def _sdpa(q, k, v, mask=None):
    """torch CPU fp64 scaled_dot_product_attention per head; q [R][Hq][d], k/v [Nk][Hq][d]."""
    tq = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]
    tk = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))[None]
    tv = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))[None]
    am = None if mask is None else torch.from_numpy(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am)
    return o[0].numpy().transpose(1, 0, 2)


def _setup(seed, hq=4, hkv=2, d=16, N=64, rows=12):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((N, hkv, d))
    V = rng.standard_normal((N, hkv, d))
    qf = rng.standard_normal((rows, hq, d))
    kf = rng.standard_normal((rows, hkv, d))
    vf = rng.standard_normal((rows, hkv, d))
    return rng, K, V, qf, kf, vf


def test_attention_identity_rotation_equals_sdpa():
    _, K, V, qf, kf, vf = _setup(6)
    N, rows, g = K.shape[0], qf.shape[0], 2
    sel = np.array([1, 2, 30, 40, 41, 63, 10, 11])
    sel.sort()
    zeros_k = np.zeros(N, dtype=np.int64)
    zeros_r = np.zeros(rows, dtype=np.int64)
    got = method.fused_attention_request(qf, kf, vf, zeros_r, K, V, zeros_k, sel, 1e4)
    keep = np.setdiff1d(np.arange(N), sel)
    k_all = np.concatenate([K[keep], kf]).repeat(g, axis=1)
    v_all = np.concatenate([V[keep], vf]).repeat(g, axis=1)
    np.testing.assert_allclose(got, _sdpa(qf, k_all, v_all), atol=1e-12)


def test_attention_general_positions_equals_masked_sdpa():
    rng, K, V, qf, kf, vf = _setup(7)
    N, rows, g, theta = K.shape[0], qf.shape[0], 2, 1e4
    kpos = np.concatenate([50 + np.arange(32), 200 + np.arange(32)])
    sel = np.sort(rng.choice(N, size=8, replace=False))
    row_pos = np.concatenate([kpos[sel], 300 + np.arange(rows - 8)])
    got = method.fused_attention_request(qf, kf, vf, row_pos, K, V, kpos, sel, theta)
    keep = np.setdiff1d(np.arange(N), sel)
    key_pos = np.concatenate([kpos[keep], row_pos])
    k_all = rot_complex(np.concatenate([K[keep], kf]), key_pos, theta).repeat(g, axis=1)
    v_all = np.concatenate([V[keep], vf]).repeat(g, axis=1)
    q_rot = rot_complex(qf, row_pos, theta)
    mask = key_pos[None, :] <= row_pos[:, None]
    np.testing.assert_allclose(got, _sdpa(q_rot, k_all, v_all, mask), atol=1e-12)


def test_full_prefill_equals_causal_sdpa():
    rng = np.random.default_rng(8)
    n, hq, hkv, d, theta = 20, 4, 1, 8, 1e4
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    pos = np.cumsum(rng.integers(1, 5, n)) + 10
    got = method.full_prefill(q, k, v, pos, theta)
    mask = np.tril(np.ones((n, n), dtype=bool))
    ref = _sdpa(rot_complex(q, pos, theta), rot_complex(k, pos, theta).repeat(hq, axis=1),
                v.repeat(hq, axis=1), mask)
    np.testing.assert_allclose(got, ref, atol=1e-12)


def _oracle_request(batch, b=0, sel=None):
    r = batch.requests[b]
    kp = batch.k_pool.to(torch.float64).numpy()
    vp = batch.v_pool.to(torch.float64).numpy()
    K, V, kpos = method.request_cached(r.spans, kp, vp)
    rb = batch.row_bases()[b]
    qb = batch.query_bases()[b]
    q = batch.q_query[qb: qb + r.n_query].to(torch.float64).numpy()
    qpos = r.query_pos0 + np.arange(r.n_query)
    imp = method.score_request(q, qpos, K, kpos, batch.theta)
    if sel is None:
        sel = method.select_topk_request(imp.astype(np.float32), [s.n_pages * 16 for s in r.spans],
                                         [s.k for s in r.spans])
    row_pos = method.row_positions(sel, kpos, r.n_query, r.query_pos0)
    qf = batch.q_fresh[rb: rb + r.n_rows].to(torch.float64).numpy()
    kf = batch.k_fresh[rb: rb + r.n_rows].to(torch.float64).numpy()
    vf = batch.v_fresh[rb: rb + r.n_rows].to(torch.float64).numpy()
    out = method.fused_attention_request(qf, kf, vf, row_pos, K, V, kpos, sel, batch.theta)
    return dict(K=K, V=V, kpos=kpos, imp=imp, sel=sel, row_pos=row_pos, qf=qf, kf=kf, vf=vf,
                out=out)


def test_full_recompute_reproduces_full_prefill():
    # every token of every span recomputed: no cached key survives
    b = small_custom_batch([(0, 2, 0, 32), (2, 1, 32, 16)], n_query=6, hq=4, hkv=2, d=16)
    o = _oracle_request(b)
    assert len(o["sel"]) == 48
    ref = method.full_prefill(o["qf"], o["kf"], o["vf"], o["row_pos"], b.theta)
    np.testing.assert_allclose(o["out"], ref, atol=1e-12)


def test_offset_reuse_matches_fresh_prefill_at_2048():
    """A span cached once (physical pages 0..1) is used at offset 0 by request 0 and at offset
    2048 by request 1; request 1 must equal a fresh computation whose keys were rotated at 2048."""
    b = small_custom_batch([(0, 2, 0, 0)], n_query=4, hq=4, hkv=2, d=16,
                           extra_requests=[([(0, 2, 2048, 0)], 4, 2048 + 32)])
    o1 = _oracle_request(b, 1)
    theta, g = b.theta, 2
    kp = b.k_pool.to(torch.float64).numpy()
    vp = b.v_pool.to(torch.float64).numpy()
    K = kp[[0, 1]].transpose(0, 2, 1, 3).reshape(32, 2, 16)
    V = vp[[0, 1]].transpose(0, 2, 1, 3).reshape(32, 2, 16)
    kpos = 2048 + np.arange(32)
    qpos = o1["row_pos"]
    k_all = np.concatenate([rot_complex(K, kpos, theta), rot_complex(o1["kf"], qpos, theta)])
    v_all = np.concatenate([V, o1["vf"]])
    mask = np.concatenate([kpos, qpos])[None, :] <= qpos[:, None]
    ref = _sdpa(rot_complex(o1["qf"], qpos, theta), k_all.repeat(g, axis=1),
                v_all.repeat(g, axis=1), mask)
    np.testing.assert_allclose(o1["out"], ref, atol=1e-12)
    # request 0 sees the same tokens shifted by -2048 and the same query: scores are unchanged
    o0 = _oracle_request(b, 0)
    q0 = b.q_query[:4].to(torch.float64).numpy()
    q1 = b.q_query[4:8].to(torch.float64).numpy()
    imp_shift = method.score_request(q1, 32 + np.arange(4), o0["K"], o0["kpos"], theta)
    np.testing.assert_allclose(o1["imp"], imp_shift, atol=1e-12)
    assert not np.allclose(q0, q1)


def test_shift_invariance_of_importance_and_output():
    b = small_custom_batch([(0, 2, 5, 6), (2, 2, 40, 5)], n_query=5, hq=4, hkv=2, d=16)
    o = _oracle_request(b)
    D = 1234
    imp2 = method.score_request(b.q_query.to(torch.float64).numpy(),
                                b.requests[0].query_pos0 + D + np.arange(5), o["K"],
                                o["kpos"] + D, b.theta)
    np.testing.assert_allclose(imp2, o["imp"], atol=1e-12)
    out2 = method.fused_attention_request(o["qf"], o["kf"], o["vf"], o["row_pos"] + D, o["K"],
                                          o["V"], o["kpos"] + D, o["sel"], b.theta)
    np.testing.assert_allclose(out2, o["out"], atol=1e-12)


def test_selection_invariance_when_fresh_equals_cached():
    """If the fresh K/V of the recomputed tokens equal their cached copies, the merged key set is
    the same for every selection, so the query rows' output does not depend on the selection."""
    b = small_custom_batch([(0, 3, 0, 8), (3, 2, 48, 4)], n_query=6, hq=4, hkv=2, d=16)
    o = _oracle_request(b)
    r = b.requests[0]
    T = r.n_query
    outs = []
    rng = np.random.default_rng(9)
    for trial in range(3):
        if trial == 0:
            sel = o["sel"]
        else:
            sel = np.sort(np.concatenate([rng.choice(48, 8, replace=False),
                                          48 + rng.choice(32, 4, replace=False)]))
        row_pos = method.row_positions(sel, o["kpos"], T, r.query_pos0)
        kf = np.concatenate([o["K"][sel], o["kf"][-T:]])
        vf = np.concatenate([o["V"][sel], o["vf"][-T:]])
        qf = np.concatenate([o["qf"][:len(sel)], o["qf"][-T:]])
        outs.append(method.fused_attention_request(qf, kf, vf, row_pos, o["K"], o["V"], o["kpos"],
                                                   sel, b.theta)[-T:])
    # no recompute at all
    row_pos = method.row_positions(np.zeros(0, dtype=np.int64), o["kpos"], T, r.query_pos0)
    outs.append(method.fused_attention_request(o["qf"][-T:], o["kf"][-T:], o["vf"][-T:], row_pos,
                                               o["K"], o["V"], o["kpos"],
                                               np.zeros(0, dtype=np.int64), b.theta))
    for x in outs[1:]:
        np.testing.assert_allclose(x, outs[0], atol=1e-12)


def test_gqa_map_equals_mha_with_repeated_kv_heads():
    rng, K, V, qf, kf, vf = _setup(10, hq=8, hkv=2)
    kpos = np.arange(64) + 3
    sel = np.array([4, 9, 33, 50])
    row_pos = np.concatenate([kpos[sel], 100 + np.arange(8)])
    a = method.fused_attention_request(qf, kf, vf, row_pos, K, V, kpos, sel, 1e4)
    rep = lambda x: x.repeat(4, axis=1)   # kv head h // 4 serves q head h
    m = method.fused_attention_request(qf, rep(kf), rep(vf), row_pos, rep(K), rep(V), kpos, sel, 1e4)
    np.testing.assert_allclose(a, m, atol=1e-13)
    q = rng.standard_normal((3, 8, 16))
    ia = method.score_request(q, 200 + np.arange(3), K, kpos, 1e4)
    im = method.score_request(q, 200 + np.arange(3), rep(K), kpos, 1e4)
    np.testing.assert_allclose(ia, im, atol=1e-12)


def test_workload_layout_invariants():
    for name, cfg in CONFIGS.items():
        for r in make_layout(cfg):
            pos_end = -1
            for s in r.spans:
                assert s.pos0 > pos_end
                pos_end = s.pos0 + s.n_pages * 16 - 1
                assert 0 <= s.k <= s.n_pages * 16
            assert r.query_pos0 > pos_end
            assert r.query_pos0 + r.n_query <= 65536
