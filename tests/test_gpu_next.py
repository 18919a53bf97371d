"""GPU parity of the variants beyond the per-span hot path: the pages' global Top-N (one budget
per request over all its cached tokens, QCFuse 2B), anchor extraction (each span's tokens with the
largest key norm, QCFuse 2A), anchor-prefixed query probing (QCFuse 2A injection / Phase 2) and the
layer-pipelined pool prefetch (QCFuse 2C / Phase 4, host tier).  Selections and copies are
bit-exact (selections when fed the oracle's fp32 values); key norms are within 1e-5 relative of
the fp64 oracle; attention outputs within 2e-2 absolute + 1e-2 relative."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import position_independent_kv_critical_gb300 as pcf
from oracle import method
from workload import CONFIGS, PAGE, make_batch, make_layout, small_custom_batch

from gpu_util import GpuBatch, assert_close_out

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-5


def _layout(cfg, reqs):
    n_phys = cfg.pool_spans * cfg.span_len // PAGE
    return pcf.Layout(reqs, cfg.hq, cfg.hkv, cfg.d, n_phys, max(r.query_pos0 + r.n_query for r in reqs) + 1)


def _run_global(L, imp):
    sel = torch.empty(max(1, L.total_sel), dtype=torch.int32, device="cuda")
    ex = torch.empty(max(1, L.total_pages), dtype=torch.int16, device="cuda")
    rp = torch.empty(max(1, L.total_rows), dtype=torch.int32, device="cuda")
    pcf.select_topn_global(L, torch.as_tensor(imp).cuda(), sel, ex, rp)
    pcf.check_device_error()
    return (sel[: L.total_sel].cpu().numpy(), ex[: L.total_pages].cpu().numpy().view(np.uint16),
            rp[: L.total_rows].cpu().numpy())


# ------------------------------------------------------------------ global Top-N

@pytest.mark.parametrize("name", list(CONFIGS))
def test_topn_global_bit_exact_planted_ties_full_size(name):
    cfg = CONFIGS[name]
    reqs = make_layout(cfg)
    L = _layout(cfg, reqs)
    rng = np.random.default_rng(cfg.seed + 7)
    imp = (rng.integers(0, 24, size=L.total_tokens) * 0.03125).astype(np.float32)
    sel, ex, rp = _run_global(L, imp)
    tb = sb = pb = rb = 0
    for r in reqs:
        exp = method.select_topn_global_request(imp[tb: tb + r.n_cached], r.n_sel)
        assert np.array_equal(sel[sb: sb + r.n_sel], exp)
        npg = r.n_cached // PAGE
        assert np.array_equal(ex[pb: pb + npg], method.exclusion_masks(exp, npg))
        kpos = np.concatenate([s.pos0 + np.arange(s.n_pages * PAGE) for s in r.spans])
        assert np.array_equal(rp[rb: rb + r.n_rows], method.row_positions(exp, kpos, r.n_query, r.query_pos0))
        tb += r.n_cached
        sb += r.n_sel
        pb += npg
        rb += r.n_rows


@pytest.mark.parametrize("ks", [(0, 0), (32, 48), (5, 0), (0, 7)])
def test_topn_global_budget_extremes(ks):
    """Budgets of nothing, of every token, and all of it drawn from one span."""
    b = small_custom_batch([(0, 2, 0, ks[0]), (4, 3, 64, ks[1])], n_query=5, n_phys_pages=8)
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, b.max_pos + 1)
    rng = np.random.default_rng(sum(ks))
    imp = rng.random(L.total_tokens).astype(np.float32)
    sel, _, _ = _run_global(L, imp)
    assert np.array_equal(sel, method.select_topn_global_request(imp, b.requests[0].n_sel))


@pytest.mark.parametrize("name", ["tiny", "llama8b_layer"])
def test_topn_global_selection_drives_the_fused_attention(name):
    """Global selection on the oracle's fp32 scores, then the fused attention over it, against the
    oracle's attention with the oracle's global selection."""
    gb = GpuBatch(make_batch(name))
    r = gb.b.requests[0]
    imp32 = gb.oracle_score(0).astype(np.float32)
    pad = np.zeros(gb.L.total_tokens, dtype=np.float32)
    pad[: r.n_cached] = imp32
    pcf.select_topn_global(gb.L, torch.as_tensor(pad).cuda(), gb.cf.sel_idx, gb.cf.excl, gb.cf.row_pos)
    pcf.check_device_error()
    sel_gpu = gb.cf.sel_idx[: r.n_sel].cpu().numpy()
    sel = method.select_topn_global_request(imp32, r.n_sel)
    assert np.array_equal(sel_gpu, sel)
    out = gb.attention()
    exp, _ = gb.oracle_attention(0, sel)
    assert_close_out(out[: r.n_rows], exp, f"{name} global Top-N attention")


# ------------------------------------------------------------------ anchors

def _norms_gpu(gb):
    norms = torch.empty(gb.L.total_tokens, dtype=torch.float32, device="cuda")
    pcf.key_norms(gb.L, gb.k_pool, norms)
    pcf.check_device_error()
    return norms


@pytest.mark.parametrize("name", ["tiny", "llama8b_layer", "concurrent_reuse"])
def test_key_norms_match_oracle(name):
    gb = GpuBatch(make_batch(name))
    got = _norms_gpu(gb).cpu().numpy()
    ids = range(len(gb.b.requests)) if name != "concurrent_reuse" else (0, 17, 31)
    for i in ids:
        r, K, _, _ = gb.oracle_request(i)
        tb = gb.tok_base[i]
        np.testing.assert_allclose(got[tb: tb + r.n_cached], method.key_norms(K), rtol=NORM_RTOL)


@pytest.mark.parametrize("name,m_pct", [("tiny", 5), ("llama8b_layer", 3), ("concurrent_reuse", 2)])
def test_anchors_bit_exact_on_oracle_norms_and_close_on_gpu_norms(name, m_pct):
    """Anchors = per-span Top-m on the key norms: a layout whose span k's are the anchor counts,
    run through pcf_select_topk; bit-exact on the oracle's fp32 norms, and (almost always) the same
    tokens from the GPU's own norms."""
    b = make_batch(name)
    reqs = [dataclasses.replace(r, spans=[dataclasses.replace(s, k=method.k_from_percent(m_pct, s.n_pages * PAGE))
                                          for s in r.spans]) for r in b.requests]
    gb = GpuBatch(dataclasses.replace(b, requests=reqs))
    oracle_norms = np.zeros(gb.L.total_tokens, dtype=np.float32)
    for i in range(len(reqs)):
        _, K, _, _ = gb.oracle_request(i)
        oracle_norms[gb.tok_base[i]: gb.tok_base[i] + K.shape[0]] = method.key_norms(K)
    sel, _, _ = gb.topk(oracle_norms)
    gpu_norms = _norms_gpu(gb)
    pcf.select_topk(gb.L, gpu_norms, gb.cf.sel_idx, gb.cf.excl, gb.cf.row_pos)
    pcf.check_device_error()
    sel_g = gb.cf.sel_idx[: gb.L.total_sel].cpu().numpy()
    same = total = 0
    for i, r in enumerate(reqs):
        lens = [s.n_pages * PAGE for s in r.spans]
        exp = method.select_anchors_request(oracle_norms[gb.tok_base[i]: gb.tok_base[i] + r.n_cached], lens,
                                            [s.k for s in r.spans])
        sb = gb.sel_base[i]
        assert np.array_equal(sel[sb: sb + r.n_sel], exp)
        same += len(np.intersect1d(sel_g[sb: sb + r.n_sel], exp))
        total += len(exp)
    assert same >= 0.99 * total, (same, total)


# ------------------------------------------------------------------ anchor-prefixed query probing

def _anchor_batch(name, pct):
    b = make_batch(name)
    reqs = [dataclasses.replace(r, spans=[dataclasses.replace(s, k=method.anchor_count(pct, s.n_pages * PAGE))
                                          for s in r.spans]) for r in b.requests]
    return dataclasses.replace(b, requests=reqs)


@pytest.mark.parametrize("name,pct,req_ids", [("tiny", 12, (0,)), ("llama8b_layer", 6, (0,)),
                                              ("concurrent_reuse", 3, (0, 13, 31))])
def test_anchor_probe_matches_oracle(name, pct, req_ids):
    """Anchors from the oracle's fp32 key norms (per span, whole pages), packed into pages of their
    own (bit-exact), then the query tokens attend over them as a prefix through the fused
    attention on a second layout; against the oracle's probe."""
    ab = _anchor_batch(name, pct)
    gb = GpuBatch(ab)
    reqs = ab.requests
    norms = np.zeros(gb.L.total_tokens, dtype=np.float32)
    for i in range(len(reqs)):
        _, K, _, _ = gb.oracle_request(i)
        norms[gb.tok_base[i]: gb.tok_base[i] + K.shape[0]] = method.key_norms(K)
    gb.topk(norms)
    A_tot = gb.L.total_sel
    ka = torch.empty((A_tot // PAGE, ab.hkv, PAGE, ab.d), dtype=torch.bfloat16, device="cuda")
    va = torch.empty_like(ka)
    pcf.pack_anchor_pages(gb.L, gb.cf.sel_idx, gb.k_pool, gb.v_pool, ka, va)
    pcf.check_device_error()
    sel = gb.cf.sel_idx[:A_tot].cpu().numpy()
    ka_rows = ka.permute(0, 2, 1, 3).reshape(A_tot, ab.hkv, ab.d).double().cpu().numpy()
    va_rows = va.permute(0, 2, 1, 3).reshape(A_tot, ab.hkv, ab.d).double().cpu().numpy()
    # the probe: one span of anchor pages per request, the query right after it
    probe = [dataclasses.replace(r, spans=[dataclasses.replace(r.spans[0], phys_first_page=gb.sel_base[i] // PAGE,
                                                               n_pages=r.n_sel // PAGE, pos0=0, k=0)],
                                 query_pos0=r.n_sel) for i, r in enumerate(reqs)]
    T = [r.n_query for r in reqs]
    g = torch.Generator().manual_seed(ab.seed + 99)
    mk = lambda h: torch.randn((sum(T), h, ab.d), generator=g).to(torch.bfloat16)
    q, k, v = mk(ab.hq), mk(ab.hkv), mk(ab.hkv)
    PL = pcf.Layout(probe, ab.hq, ab.hkv, ab.d, A_tot // PAGE, max(r.n_sel + r.n_query for r in reqs) + 1)
    rope = pcf.rope_table(ab.d, ab.theta, max(r.n_sel + r.n_query for r in reqs) + 1).cuda()
    pcf_cf = pcf.CacheFusion(PL, rope, row_elems=0)
    pcf.select_topk(PL, torch.zeros(max(1, PL.total_tokens), dtype=torch.float32, device="cuda"),
                    pcf_cf.sel_idx, pcf_cf.excl, pcf_cf.row_pos)
    pcf.fused_attention(PL, q.cuda(), k.cuda(), v.cuda(), ka, va, pcf_cf.excl, pcf_cf.row_pos, rope,
                        pcf_cf.out, pcf_cf.ws_attn)
    pcf.check_device_error()
    out = pcf_cf.out[: PL.total_rows].float().cpu().numpy()
    qb = np.concatenate([[0], np.cumsum(T)])
    for i in req_ids:
        r = reqs[i]
        sb = gb.sel_base[i]
        _, K, V, _ = gb.oracle_request(i)
        exp_sel = method.select_anchors_request(norms[gb.tok_base[i]: gb.tok_base[i] + r.n_cached],
                                                [s.n_pages * PAGE for s in r.spans], [s.k for s in r.spans])
        assert np.array_equal(sel[sb: sb + r.n_sel], exp_sel)
        assert np.array_equal(ka_rows[sb: sb + r.n_sel], K[exp_sel])
        assert np.array_equal(va_rows[sb: sb + r.n_sel], V[exp_sel])
        sl = slice(qb[i], qb[i + 1])
        exp = method.anchor_probe_request(q[sl].double().numpy(), k[sl].double().numpy(), v[sl].double().numpy(),
                                          K[exp_sel], V[exp_sel], ab.theta)
        assert_close_out(out[sl], exp, f"{name} anchor probe request {i}")


# ------------------------------------------------------------------ layer-pipelined pool prefetch

def test_prefetch_copies_exactly_the_referenced_pages():
    """32 requests over a shared pool: every page some span references arrives (once), the others
    keep what the device pool held."""
    b = make_batch("concurrent_reuse")
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, b.max_pos + 1)
    hk, hv = b.k_pool.pin_memory(), b.v_pool.pin_memory()
    dk = torch.full_like(b.k_pool, 7.0, device="cuda")
    dv = torch.full_like(b.v_pool, 7.0, device="cuda")
    pcf.prefetch_pool_pages(L, hk, hv, dk, dv)
    torch.cuda.synchronize()
    used = np.zeros(b.n_phys_pages, dtype=bool)
    for r in b.requests:
        for s in r.spans:
            used[s.phys_first_page: s.phys_first_page + s.n_pages] = True
    assert used.any() and not used.all()
    gk, gv = dk.cpu(), dv.cpu()
    u = torch.as_tensor(used)
    assert torch.equal(gk[u].view(torch.int16), b.k_pool[u].view(torch.int16))
    assert torch.equal(gv[u].view(torch.int16), b.v_pool[u].view(torch.int16))
    assert bool((gk[~u] == 7.0).all()) and bool((gv[~u] == 7.0).all())


def test_two_layer_pipeline_matches_resident_pools():
    """Layer 1's pool streams in from pinned host memory on a copy stream while layer 0's fused
    attention runs; each layer's output equals the one computed with its pool already resident."""
    gb = GpuBatch(make_batch("llama8b_layer"))
    b = gb.b
    g = torch.Generator().manual_seed(b.seed + 123)
    host_k = [b.k_pool, torch.randn(b.k_pool.shape, generator=g).to(torch.bfloat16)]
    host_v = [b.v_pool, torch.randn(b.v_pool.shape, generator=g).to(torch.bfloat16)]
    host_k = [t.pin_memory() for t in host_k]
    host_v = [t.pin_memory() for t in host_v]
    gb.score()
    gb.topk()
    ref = []
    for l in range(2):
        gb.k_pool, gb.v_pool = host_k[l].cuda(), host_v[l].cuda()
        ref.append(gb.attention().copy())
    dk = [torch.empty_like(host_k[0], device="cuda") for _ in range(2)]
    dv = [torch.empty_like(host_v[0], device="cuda") for _ in range(2)]
    copy = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    with torch.cuda.stream(copy):
        pcf.prefetch_pool_pages(gb.L, host_k[0], host_v[0], dk[0], dv[0], stream=copy)
        ready[0].record(copy)
    outs = []
    for l in range(2):
        torch.cuda.current_stream().wait_event(ready[l])
        if l + 1 < 2:
            with torch.cuda.stream(copy):
                pcf.prefetch_pool_pages(gb.L, host_k[l + 1], host_v[l + 1], dk[l + 1], dv[l + 1], stream=copy)
                ready[l + 1].record(copy)
        gb.k_pool, gb.v_pool = dk[l], dv[l]
        outs.append(gb.attention().copy())
    for l in range(2):
        assert np.array_equal(outs[l], ref[l]), l


# ------------------------------------------------------------------ all-layer importance (QCAll)

@pytest.mark.parametrize("name,n_layers", [("tiny", 3), ("llama8b_layer", 4), ("long_context", 4)])
def test_all_layer_importance_matches_oracle(name, n_layers):
    from workload import layer_inputs
    b = make_batch(name)
    gb = GpuBatch(b)
    qs, ks = layer_inputs(b, n_layers)
    qd = [t.cuda() for t in qs]
    kd = [t.cuda() for t in ks]
    n = gb.L.total_tokens
    per = torch.full((n_layers, n), float("nan"), dtype=torch.float32, device="cuda")
    tot = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    pcf.score_layers(gb.L, qd, kd, gb.rope, per, tot, gb.cf.ws_score)
    pcf.check_device_error()
    per_h, tot_h = per.cpu().numpy(), tot.cpu().numpy()
    # the sum is the layers' fp32 values added in layer order
    acc = per_h[0].copy()
    for l in range(1, n_layers):
        acc += per_h[l]
    assert np.array_equal(tot_h, acc)
    r = b.requests[0]
    K_l, kpos = [], None
    for k in ks:
        K, _, kpos = method.request_cached(r.spans, k.double().numpy(), b.v_pool.double().numpy())
        K_l.append(K)
    qpos = r.query_pos0 + np.arange(r.n_query)
    exp_per, exp_tot = method.score_layers_request([q.double().numpy() for q in qs], qpos, K_l, kpos, b.theta)
    for l in range(n_layers):
        err = np.abs(per_h[l, : r.n_cached] - exp_per[l])
        assert np.all(err <= 1e-3 * np.abs(exp_per[l]) + 1e-7), f"layer {l}: max rel {(err / exp_per[l]).max():.2e}"
    err = np.abs(tot_h[: r.n_cached] - exp_tot)
    assert np.all(err <= 1e-3 * np.abs(exp_tot) + 1e-7)
    # layer 0 is the critical-layer call itself
    assert np.array_equal(per_h[0], gb.score())


def test_all_layer_importance_of_one_layer_is_the_critical_layer_score():
    b = make_batch("llama8b_layer")
    gb = GpuBatch(b)
    n = gb.L.total_tokens
    per = torch.empty((1, n), dtype=torch.float32, device="cuda")
    tot = torch.empty((n,), dtype=torch.float32, device="cuda")
    pcf.score_layers(gb.L, [gb.q_query], [gb.k_pool], gb.rope, per, tot, gb.cf.ws_score)
    pcf.check_device_error()
    one = gb.score()
    assert np.array_equal(per[0].cpu().numpy(), one) and np.array_equal(tot.cpu().numpy(), one)
