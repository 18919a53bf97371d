"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Tolerances (stated for this path): fp32 importance within 1e-3 relative; bf16 attention output
within 2e-2 absolute + 1e-2 relative; top-k, exclusion bits, row positions and the gather are
bit-exact.  Top-k is fed the oracle's scores; the attention is fed the oracle's selection, so
near-ties in the GPU scores cannot change which keys the attention sees.  Large workloads run in
their full launch configuration and are checked on sampled requests / rows.
"""
import numpy as np
import pytest
import torch

import position_independent_kv_critical_gb300 as pcf
from oracle import method
from workload import CONFIGS, PAGE, hidden_rows, make_batch, make_layout, small_custom_batch

from gpu_util import GpuBatch, assert_close_imp, assert_close_out

pytestmark = pytest.mark.gpu

_cache = {}


def gpu_batch(name, pct=None):
    key = (name, pct)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        _cache[key] = GpuBatch(make_batch(name, pct))
    return _cache[key]


def _sample_rows(n_rows, n_sel, k=48):
    rows = set(range(min(8, n_rows)))
    rows |= set(range(max(0, n_sel - 4), min(n_rows, n_sel + 4)))
    rows |= set(range(max(0, n_rows - 12), n_rows))
    rng = np.random.default_rng(n_rows)
    rows |= set(rng.choice(n_rows, size=min(n_rows, k), replace=False).tolist())
    return np.array(sorted(rows))


def check_batch(gb: GpuBatch, req_ids=None, sample_rows=False, imp_only_ids=(), paged=False):
    """Importance, top-k and attention of the requests `req_ids` (all by default) against the
    oracle; `imp_only_ids` are further requests whose importance alone is compared; `paged` runs
    scoring and the attention through pcf_score_paged and pcf_fused_attention_paged."""
    b = gb.b
    ids = list(range(len(b.requests))) if req_ids is None else list(req_ids)
    # 1) importance
    got_imp = gb.score(paged=paged)
    for i in imp_only_ids:
        r = b.requests[i]
        t0 = gb.tok_base[i]
        assert_close_imp(got_imp[t0: t0 + r.n_cached], gb.oracle_score(i), f"importance req {i}")
    imps = {}
    for i in ids:
        r = b.requests[i]
        exp = gb.oracle_score(i)
        t0 = gb.tok_base[i]
        assert_close_imp(got_imp[t0: t0 + r.n_cached], exp, f"importance req {i}")
        imps[i] = exp.astype(np.float32)
    # 2) top-k bit-exact on the oracle's scores (other requests: their GPU scores)
    feed = got_imp.copy()
    for i in ids:
        feed[gb.tok_base[i]: gb.tok_base[i] + b.requests[i].n_cached] = imps[i]
    sel, excl, row_pos = gb.topk(feed)
    sels = []
    for i, r in enumerate(b.requests):
        s0 = gb.sel_base[i]
        sels.append(sel[s0: s0 + r.n_sel].astype(np.int64))
    for i in ids:
        exp_sel = gb.oracle_select(i, imps[i])
        assert np.array_equal(sels[i], exp_sel), f"top-k req {i}"
    exp_excl, exp_rp = gb.selection_inputs(sels)
    assert np.array_equal(excl, exp_excl)
    assert np.array_equal(row_pos, exp_rp)
    # 3) attention with the oracle's selection
    out = gb.attention(exp_excl, exp_rp, paged=paged)
    for i in ids:
        r = b.requests[i]
        rows = _sample_rows(r.n_rows, r.n_sel) if sample_rows else None
        exp, _ = gb.oracle_attention(i, sels[i], rows=rows)
        rb = gb.row_base[i]
        got = out[rb: rb + r.n_rows]
        got = got if rows is None else got[rows]
        assert_close_out(got, exp, f"attention req {i}")


# ------------------------------------------------------------------ the five workloads

def test_tiny_full():
    check_batch(gpu_batch("tiny"))


def test_llama8b_layer_full():
    check_batch(gpu_batch("llama8b_layer"))


def test_concurrent_reuse_sampled():
    check_batch(gpu_batch("concurrent_reuse"), req_ids=[0, 7, 31], sample_rows=True)


@pytest.mark.parametrize("pct", [5, 10, 15, 20, 30])
def test_long_context_sweep_sampled(pct):
    check_batch(gpu_batch("long_context", pct), sample_rows=True)


def _heaviest_span_requests(b, n=2):
    """Requests holding the physical spans that the Zipf draws reference most often."""
    refs = {}
    for i, r in enumerate(b.requests):
        for s in r.spans:
            refs.setdefault(s.phys_first_page, []).append(i)
    top = sorted(refs.items(), key=lambda kv: (-len(kv[1]), kv[0]))[:n]
    return [reqs[len(reqs) // 2] for _, reqs in top]


def test_batch70b_sampled():
    gb = gpu_batch("batch70b")
    spread = list(range(0, 64, 9))                     # 0, 9, ..., 63: eight requests over the batch
    extra = [i for i in spread + _heaviest_span_requests(gb.b) if i not in (0, 63)]
    check_batch(gb, req_ids=[0, 63], sample_rows=True, imp_only_ids=sorted(set(extra)))


# ------------------------------------------------------------------ top-k at full size, planted ties

@pytest.mark.parametrize("name", list(CONFIGS))
def test_topk_bit_exact_planted_ties_full_size(name):
    cfg = CONFIGS[name]
    reqs = make_layout(cfg)
    n_phys = cfg.pool_spans * cfg.span_len // PAGE
    L = pcf.Layout(reqs, cfg.hq, cfg.hkv, cfg.d, n_phys, max(r.query_pos0 + r.n_query for r in reqs) + 1)
    rng = np.random.default_rng(cfg.seed)
    imp = (rng.integers(0, 24, size=L.total_tokens) * 0.03125).astype(np.float32)
    dev_imp = torch.as_tensor(imp).cuda()
    sel = torch.empty(L.total_sel, dtype=torch.int32, device="cuda")
    ex = torch.empty(L.total_pages, dtype=torch.int16, device="cuda")
    rp = torch.empty(L.total_rows, dtype=torch.int32, device="cuda")
    pcf.select_topk(L, dev_imp, sel, ex, rp)
    pcf.check_device_error()
    sel = sel.cpu().numpy()
    tb = sb = 0
    for r in reqs:
        exp = method.select_topk_request(imp[tb: tb + r.n_cached], [s.n_pages * 16 for s in r.spans],
                                         [s.k for s in r.spans])
        assert np.array_equal(sel[sb: sb + r.n_sel], exp)
        tb += r.n_cached
        sb += r.n_sel


# ------------------------------------------------------------------ gather

@pytest.mark.parametrize("name", ["tiny", "llama8b_layer"])
def test_gather_bit_exact(name):
    gb = gpu_batch(name)
    D = gb.b.hq * gb.b.d
    src = hidden_rows(torch.arange(gb.L.total_tokens, device="cuda"), D)
    gb.score()
    sel, _, _ = gb.topk()
    dst = torch.empty((gb.L.total_sel, D), dtype=torch.bfloat16, device="cuda")
    pcf.gather_rows(gb.L, gb.cf.sel_idx, src, dst)
    pcf.check_device_error()
    glob = np.concatenate([gb.tok_base[i] + sel[gb.sel_base[i]: gb.sel_base[i] + r.n_sel]
                           for i, r in enumerate(gb.b.requests)])
    exp = method.gather_rows(hidden_rows(torch.arange(gb.L.total_tokens), D).view(torch.int16).numpy(), glob)
    assert np.array_equal(dst.cpu().view(torch.int16).numpy(), exp)


def test_gpu_scores_to_gpu_topk_overlap():
    gb = gpu_batch("llama8b_layer")
    gb.score()
    sel, _, _ = gb.topk()
    exp = gb.oracle_select(0, gb.oracle_score(0).astype(np.float32))
    overlap = len(np.intersect1d(sel, exp)) / len(exp)
    assert overlap >= 0.99, overlap


def test_score_is_deterministic():
    gb = gpu_batch("llama8b_layer")
    a = gb.score().copy()
    b = gb.score().copy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_step_from_host_matches_device_step():
    """The pipelined host-input step (uploads and downloads on their own streams, two input slots)
    gives bit for bit the device step's O and selection, with four steps on two different input
    sets issued back to back before any of them is waited for."""
    b = make_batch("llama8b_layer")
    mp = b.max_pos + 1
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, mp)
    rope = pcf.rope_table(b.d, b.theta, mp).cuda()
    cf = pcf.CacheFusion(L, rope)
    k_pool, v_pool = b.k_pool.cuda(), b.v_pool.cuda()
    sets = [(b.q_query, b.q_fresh, b.k_fresh, b.v_fresh),
            ((b.q_query.float() * -0.75).to(torch.bfloat16), (b.q_fresh.float() * 0.5).to(torch.bfloat16),
             b.k_fresh.flip(0).contiguous(), (b.v_fresh.float() * -1.0).to(torch.bfloat16))]
    refs = []
    for qq, qf, kf, vf in sets:
        out = cf.step(qq.cuda(), k_pool, v_pool, qf.cuda(), kf.cuda(), vf.cuda())
        refs.append((out.cpu().clone(), cf.sel_idx.cpu().clone()))
    torch.cuda.synchronize()
    host = [[t.pin_memory() for t in st] for st in sets]
    outs = [torch.zeros_like(cf.out, device="cpu").pin_memory() for _ in range(4)]
    sels = [torch.zeros_like(cf.sel_idx, device="cpu").pin_memory() for _ in range(4)]
    for k in range(4):
        cf.step_from_host(*host[k % 2], k_pool, v_pool, outs[k], sels[k])
    cf.wait_host_results()
    torch.cuda.synchronize()
    pcf.check_device_error()
    for k in range(4):
        ref_out, ref_sel = refs[k % 2]
        assert torch.equal(outs[k].view(torch.int16), ref_out.view(torch.int16)), k
        assert torch.equal(sels[k], ref_sel), k


def test_attention_is_deterministic_under_dynamic_item_order():
    """The persistent attention kernel hands items to CTAs in whatever order they free up; each
    item's rows (or partial slot) are written by whichever CTA runs it, so two runs must agree
    bit for bit (long context: about four items per CTA, no key-range splits; Llama-8B layer:
    split items merged afterwards)."""
    for name in ("llama8b_layer", "long_context"):
        gb = gpu_batch(name)
        gb.score()
        gb.topk()
        a = gb.attention().copy()
        b = gb.attention().copy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), name


# ------------------------------------------------------------------ scenarios from the pages

def test_offset_0_and_2048_share_physical_pages():
    """MiniPIC 1 / 2.1: one physical span serves a request at offset 0 and one at 2048."""
    b = small_custom_batch([(0, 8, 0, 20)], n_query=16, hq=8, hkv=2, d=128, theta=5e5,
                           extra_requests=[([(0, 8, 2048, 20)], 16, 2048 + 128)])
    check_batch(GpuBatch(b))


def test_full_recompute_equals_full_prefill():
    b = small_custom_batch([(0, 4, 0, 64), (4, 3, 64, 48)], n_query=9, hq=8, hkv=2, d=128, theta=5e5)
    gb = GpuBatch(b)
    r = b.requests[0]
    sel = np.arange(r.n_cached)
    excl, row_pos = gb.selection_inputs([sel])
    out = gb.attention(excl, row_pos)
    exp = method.full_prefill(b.q_fresh.double().numpy(), b.k_fresh.double().numpy(),
                              b.v_fresh.double().numpy(), row_pos.astype(np.int64), b.theta)
    assert_close_out(out, exp, "100% recompute")


def test_fresh_equal_cached_gives_no_recompute_attention():
    b = small_custom_batch([(0, 6, 0, 30), (6, 5, 100, 25)], n_query=12, hq=8, hkv=2, d=128, theta=5e5)
    r = b.requests[0]
    gb = GpuBatch(b)
    rng = np.random.default_rng(3)
    sel = np.sort(np.concatenate([rng.choice(96, 30, replace=False), 96 + rng.choice(80, 25, replace=False)]))
    pages = [s.phys_first_page + i for s in r.spans for i in range(s.n_pages)]
    kc = b.k_pool[pages].permute(0, 2, 1, 3).reshape(-1, b.hkv, b.d)
    vc = b.v_pool[pages].permute(0, 2, 1, 3).reshape(-1, b.hkv, b.d)
    gb.k_fresh[: len(sel)] = kc[sel].cuda()
    gb.v_fresh[: len(sel)] = vc[sel].cuda()
    excl, row_pos = gb.selection_inputs([sel])
    out = gb.attention(excl, row_pos)[-r.n_query:]
    _, K, V, kpos = gb.oracle_request(0)
    qpos = method.row_positions(np.zeros(0, dtype=np.int64), kpos, r.n_query, r.query_pos0)
    exp = method.fused_attention_request(b.q_fresh[-r.n_query:].double().numpy(),
                                         b.k_fresh[-r.n_query:].double().numpy(),
                                         b.v_fresh[-r.n_query:].double().numpy(), qpos, K, V, kpos,
                                         np.zeros(0, dtype=np.int64), b.theta)
    assert_close_out(out, exp, "fresh == cached")


@pytest.mark.parametrize("case", [
    dict(spans=[(0, 1, 0, 0)], n_query=1),                         # one page, nothing recomputed, T=1
    dict(spans=[(0, 2, 5, 32)], n_query=3),                        # k = L
    dict(spans=[(0, 3, 0, 1), (3, 5, 48, 7), (8, 1, 200, 16)], n_query=7),   # ragged spans
    dict(spans=[], n_query=5),                                     # no cached spans at all
    dict(spans=[(0, 9, 0, 30)], n_query=0),                        # no query rows
])
@pytest.mark.parametrize("shape", [dict(hq=4, hkv=4, d=64), dict(hq=16, hkv=2, d=128),
                                   dict(hq=8, hkv=2, d=64)])
def test_edge_cases(case, shape):
    b = small_custom_batch(case["spans"], case["n_query"], n_phys_pages=12, theta=1e4, **shape)
    check_batch(GpuBatch(b))


@pytest.mark.parametrize("shape", [dict(hq=12, hkv=3, d=128), dict(hq=24, hkv=12, d=64)])
def test_head_counts_not_multiples_of_eight(shape):
    """The rotation kernels stage tiles of up to 8 heads: 12 query heads make a full group and a
    group of 4, 12 kv heads the same for the cached keys' pages, and 3 kv heads one short page
    group; ragged spans and a query count that is not a multiple of 16 rows."""
    b = small_custom_batch([(0, 3, 0, 5), (3, 5, 48, 19), (8, 2, 300, 0)], 21, n_phys_pages=12,
                           theta=1e4, **shape)
    check_batch(GpuBatch(b))
    check_batch(GpuBatch(b), paged=True)


def test_mixed_requests_in_one_batch():
    b = small_custom_batch([(0, 3, 7, 5)], n_query=2, hq=8, hkv=2, d=128, theta=5e5, n_phys_pages=40,
                           extra_requests=[([(3, 17, 100, 40), (20, 9, 2000, 3)], 33, 3000),
                                           ([], 4, 10),
                                           ([(0, 3, 9000, 48), (29, 11, 9100, 100)], 130, 9400)])
    check_batch(GpuBatch(b))


@pytest.mark.parametrize("name,scale", [("tiny", 8.0), ("llama8b_layer", 64.0)])
def test_large_magnitude_keys_and_queries(name, scale):
    # cached and fresh keys `scale` times the unit scale, queries divided by it (powers of two, so
    # both are exact in bf16): the rotated fp16 operands sit far from 1 -- keys up to a few hundred,
    # query elements down into fp16's subnormal range -- while every logit, hence the softmax and
    # the tolerances, stays that of the unit-scale workload.  (Scaling both up would multiply the
    # logits by scale^2, and the fp16 rounding error of a logit grows with its magnitude.)
    import dataclasses
    b = make_batch(name)
    up = lambda t: (t.float() * scale).to(torch.bfloat16)
    down = lambda t: (t.float() / scale).to(torch.bfloat16)
    check_batch(GpuBatch(dataclasses.replace(b, k_pool=up(b.k_pool), k_fresh=up(b.k_fresh),
                                             q_query=down(b.q_query), q_fresh=down(b.q_fresh))))


def test_fp16_range_overflow_is_reported_not_clamped():
    import dataclasses
    b = make_batch("tiny")
    k = b.k_pool.clone()
    page = b.requests[0].spans[2].phys_first_page
    k[page, 1, 5, 3] = 2.0e5          # one cached key element far beyond the fp16 range
    gb = GpuBatch(dataclasses.replace(b, k_pool=k))
    pcf.score(gb.L, gb.q_query, gb.k_pool, gb.rope, gb.cf.importance, gb.cf.ws_score)
    with pytest.raises(pcf.PcfError) as e:
        pcf.check_device_error()
    assert e.value.status == -8           # PCF_ERR_DEVICE_RANGE
    pcf.check_device_error()              # the word was cleared: the next check is clean
    gb_ok = GpuBatch(b)
    assert_close_imp(gb_ok.score()[: b.requests[0].n_cached], gb_ok.oracle_score(0), "after a range error")


def test_device_error_word_clean_after_runs():
    pcf.check_device_error()
