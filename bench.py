"""Benchmark of the cache-fusion hot path at the critical layer on GB300.

One step = score (query -> cached keys, each key rotated to its request's position at use time)
+ per-span top-k + gather of the recompute rows + fused attention of recomputed and query rows
over cached-minus-selected plus fresh KV, on one batch of synthetic input already resident in HBM.
The default workload is the largest single-GPU one, the 70B-shaped batch of 64 requests.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--pct P] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own shard of requests, a batch
of the workload's shape drawn with the rank's own seed (no exchange: weak scaling); the time is
the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import CONFIGS, PAGE, Request, Span, hidden_rows, make_batch  # noqa: E402

METRIC = "fused-prefill tokens/s per layer; attention TFLOP/s vs GB300 bf16 tensor peak"
DESCR = {
    "tiny": "1 request, 4 spans x 128 cached tokens + 32 query tokens, 8q/2kv heads, d=64, theta 1e4",
    "llama8b_layer": "Llama-3-8B-shaped layer: 1 request, 8 spans x 512 cached tokens (random offset) "
                     "+ 64 query tokens, 32q/8kv heads, d=128, page 16, theta 5e5",
    "concurrent_reuse": "32 requests x 10 spans (Zipf 1.1 over a pool of 64 x 1024-token spans) + 64 query "
                        "tokens, 32q/8kv, d=128",
    "long_context": "1 request, 64 spans x 512 = 32768 cached tokens + 128 query tokens, 32q/8kv, d=128",
    "batch70b": "64 requests x 16 spans x 1024 tokens (Zipf 1.0, pool 256 spans) + 128 query tokens, "
                "64q/8kv, d=128",
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def _kernel_sources_sha256():
    import hashlib
    csrc = os.path.join(ROOT, "position_independent_kv_critical_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(f.encode())
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()


def _recorded_traffic(workload):
    """DRAM bytes per launch of the fused attention from the last ncu capture, if that capture
    was taken on the same workload and the kernel sources have not changed since (else None)."""
    p = os.path.join(ROOT, "profiles", f"traffic_attn_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        rec = json.load(fh)
    if rec.get("kernel_sources_sha256") != _kernel_sources_sha256():
        return None
    return rec.get("traffic_bytes_per_launch")


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(ms: float, world: int, dev) -> float:
    """The slowest rank's step time (each rank runs its own copy of the workload: weak scaling)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _job_throughput(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job tokens/s: every rank processed its workload within the slowest rank's time."""
    return world * tokens_per_rank / (ms / 1e3)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def attention_flops(b, sel, row_pos, d, hq):
    """Algorithmic attention flops 4*d*Hq*sum_rows |visible keys| (excluded cached copies of
    recomputed tokens are not counted)."""
    total = 0
    tb = sb = rb = 0
    for r in b.requests:
        kpos = (np.concatenate([s.pos0 + np.arange(s.n_pages * 16) for s in r.spans])
                if r.spans else np.zeros(0, dtype=np.int64))
        keep = np.ones(len(kpos), dtype=bool)
        keep[sel[sb: sb + r.n_sel]] = False
        rp = row_pos[rb: rb + r.n_rows]
        keys = np.sort(np.concatenate([kpos[keep], rp]))
        total += int(np.searchsorted(keys, rp, side="right").sum())
        tb += r.n_cached
        sb += r.n_sel
        rb += r.n_rows
    return 4.0 * d * hq * total


def oracle_prepare(b):
    kp = b.k_pool.double().numpy()
    vp = b.v_pool.double().numpy()
    return dict(kp=kp, vp=vp, qq=b.q_query.double().numpy(), qf=b.q_fresh.double().numpy(),
                kf=b.k_fresh.double().numpy(), vf=b.v_fresh.double().numpy())


def oracle_step(b, prep, req_ids, row_stride=1, head_div=1):
    """The fp64 oracle on the given requests: score, per-span top-k, gather, fused attention.
    With row_stride > 1 the attention runs on every row_stride-th row only and its time counts
    row_stride times (rows spread evenly over the causal order, so the estimate is unbiased); with
    head_div > 1 everything runs on the first Hkv / head_div kv heads and their query heads (a
    problem of the same shape with fewer heads) and its time counts head_div times.
    Returns (tokens processed, seconds of oracle work those tokens take, wall seconds outside the
    attention, wall seconds of the sampled attention)."""
    from oracle import method
    qb, rb = b.query_bases(), b.row_bases()
    hk = b.hkv // head_div
    hq = hk * (b.hq // b.hkv)
    kp, vp = prep["kp"][:, :hk], prep["vp"][:, :hk]
    tokens, secs, w_fixed, w_attn = 0, 0.0, 0.0, 0.0
    for i in req_ids:
        t0 = time.perf_counter()
        r = b.requests[i]
        K, V, kpos = method.request_cached(r.spans, kp, vp)
        q = prep["qq"][qb[i]: qb[i] + r.n_query, :hq]
        imp = method.score_request(q, r.query_pos0 + np.arange(r.n_query), K, kpos, b.theta)
        sel = method.select_topk_request(imp.astype(np.float32), [s.n_pages * 16 for s in r.spans],
                                         [s.k for s in r.spans])
        method.gather_rows(np.arange(r.n_cached), sel)
        row_pos = method.row_positions(sel, kpos, r.n_query, r.query_pos0)
        t1 = time.perf_counter()
        sl = slice(rb[i], rb[i] + r.n_rows)
        method.fused_attention_request(prep["qf"][sl, :hq], prep["kf"][sl, :hk], prep["vf"][sl, :hk], row_pos, K, V,
                                       kpos, sel, b.theta, rows=np.arange(0, r.n_rows, row_stride))
        t2 = time.perf_counter()
        secs += head_div * ((t1 - t0) + row_stride * (t2 - t1))
        w_fixed += t1 - t0
        w_attn += t2 - t1
        tokens += r.n_cached + r.n_query
    return tokens, secs, w_fixed, w_attn


def _oracle_sample(b):
    """Requests and attention row stride of the base oracle sample (a few seconds of CPU work
    per step): whole small workloads; one request of the large ones with the attention on every
    16th row (the attention over a 16k-token request takes the fp64 oracle most of a minute)."""
    n = len(b.requests)
    if b.cfg_name in ("tiny", "llama8b_layer"):
        return list(range(n)), 1
    return [0], 16


def _fit_sample(b, ids, stride, w_fixed, w_attn, budget_s):
    """Coarsen the sample until one step is estimated to take at most budget_s of wall time: first
    a sparser attention row sample (at least 16 rows a request), then fewer heads."""
    max_stride = max(1, min(b.requests[i].n_rows for i in ids) // 16)
    s, h = stride, 1
    def est(s2, h2):
        return (w_fixed + w_attn * stride / s2) / h2
    while est(s, h) > budget_s:
        if s * 2 <= max_stride:
            s *= 2
        elif b.hkv % (h * 2) == 0:
            h *= 2
        else:
            break
    return s, h


def _sample_text(b, ids, stride, head_div=1):
    s = f"{len(ids)} of {len(b.requests)} requests of the {b.cfg_name} workload"
    if stride > 1:
        s += f", attention on every {stride}th row with its time counted {stride}x"
    if head_div > 1:
        s += f", {b.hkv // head_div} of {b.hkv} kv heads (and their query heads) with the time counted {head_div}x"
    return s


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    b = make_batch(args.config, args.pct)
    prep = oracle_prepare(b)
    ids, stride = _oracle_sample(b)
    # the whole --steps K --warmup W run is kept to about three minutes: the first warm-up step
    # (an extra one if W = 0) measures the base sample, and the rest use a sample coarsened to fit
    budget = 180.0 / max(1, args.steps + args.warmup)
    _, _, w_fixed, w_attn = oracle_step(b, prep, ids, stride)
    stride, hdiv = _fit_sample(b, ids, stride, w_fixed, w_attn, budget)
    for _ in range(max(0, args.warmup - 1)):
        oracle_step(b, prep, ids, stride, hdiv)
    tokens, dt = 0, 0.0
    for _ in range(args.steps):
        tk, sec, _, _ = oracle_step(b, prep, ids, stride, hdiv)
        tokens += tk
        dt += sec
    value = tokens / dt
    cores = len(os.sched_getaffinity(0))
    sample = (f"{_sample_text(b, ids, stride, hdiv)} per step (score + top-k + gather + fused attention, "
              f"fp64 NumPy, BLAS threads = all cores)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.config}: {DESCR[args.config]}"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def _anchor_probe_setup(args, pcf, b, k_pool, dev):
    """Offline: key norms, per-span anchors (whole pages) and their packed pages; online (the timed
    call): the query tokens attend over their request's anchors as a prefix (positions 0..A-1, the
    query at A..A+T-1).  Returns the timed call, its algorithmic flops and a timer of the offline
    pass."""
    import dataclasses
    v_pool = b.v_pool.to(dev)
    count = lambda n: PAGE * (-((-args.anchor_pct * n) // (100 * PAGE)))   # whole pages per span
    reqs = [dataclasses.replace(r, spans=[dataclasses.replace(s, k=count(s.n_pages * PAGE)) for s in r.spans])
            for r in b.requests]
    AL = pcf.Layout(reqs, b.hq, b.hkv, b.d, b.n_phys_pages, b.max_pos + 1, device=str(dev))
    n_anchor = AL.total_sel
    norms = torch.empty(max(1, AL.total_tokens), dtype=torch.float32, device=dev)
    sel = torch.empty(max(1, n_anchor), dtype=torch.int32, device=dev)
    ex = torch.empty(max(1, AL.total_pages), dtype=torch.int16, device=dev)
    rp = torch.empty(max(1, AL.total_rows), dtype=torch.int32, device=dev)
    ka = torch.empty((max(1, n_anchor // PAGE), b.hkv, PAGE, b.d), dtype=torch.bfloat16, device=dev)
    va = torch.empty_like(ka)

    def offline_pass():
        pcf.key_norms(AL, k_pool, norms)
        pcf.select_topk(AL, norms, sel, ex, rp)
        pcf.pack_anchor_pages(AL, sel, k_pool, v_pool, ka, va)

    offline_pass()
    sel_base = np.concatenate([[0], np.cumsum([r.n_sel for r in reqs])])
    probe = [dataclasses.replace(r, spans=[dataclasses.replace(r.spans[0], phys_first_page=int(sel_base[i]) // PAGE,
                                                               n_pages=r.n_sel // PAGE, pos0=0, k=0)],
                                 query_pos0=r.n_sel) for i, r in enumerate(reqs)]
    mp = max(r.n_sel + r.n_query for r in reqs) + 1
    PL = pcf.Layout(probe, b.hq, b.hkv, b.d, max(1, n_anchor // PAGE), mp, device=str(dev))
    rope = pcf.rope_table(b.d, b.theta, mp).to(dev)
    pcf_cf = pcf.CacheFusion(PL, rope, row_elems=0, device=str(dev))
    pcf.select_topk(PL, torch.zeros(max(1, PL.total_tokens), dtype=torch.float32, device=dev),
                    pcf_cf.sel_idx, pcf_cf.excl, pcf_cf.row_pos)
    g = torch.Generator().manual_seed(b.seed + 99)
    T = sum(r.n_query for r in reqs)
    q = b.q_query.to(dev)
    k = torch.randn((T, b.hkv, b.d), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((T, b.hkv, b.d), generator=g).to(torch.bfloat16).to(dev)
    # every query token sees its request's anchors and the query tokens up to itself
    flops = float(sum(4 * b.d * b.hq * (r.n_query * r.n_sel + r.n_query * (r.n_query + 1) // 2) for r in reqs))

    def call():
        pcf.fused_attention(PL, q, k, v, ka, va, pcf_cf.excl, pcf_cf.row_pos, rope, pcf_cf.out, pcf_cf.ws_attn)

    def time_offline():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        offline_pass()
        e1.record()
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1)

    hw = PL.host.numpy()   # compaction scan (cached pages), rotation, attention, split merge (layout word 33)
    launches = (1 if PL.total_pages else 0) + 2 + (1 if hw[33] > 0 else 0)
    return call, flops, time_offline, launches


def run_layer_prefetch(args, pcf, b, L, cf, k_pool, dev, rank, local):
    """Layers whose pools live in pinned host memory: layer l+1's referenced pages stream in on a
    copy stream (pcf_prefetch_pool_pages) while layer l's fused attention runs on two alternating
    device pools.  Reports the time per layer pipelined, and the attention and the copies alone."""
    n_layers = 4
    g = torch.Generator().manual_seed(b.seed + 321)
    host = [(b.k_pool, b.v_pool)] + [(torch.randn(b.k_pool.shape, generator=g).to(torch.bfloat16),
                                      torch.randn(b.v_pool.shape, generator=g).to(torch.bfloat16))
                                     for _ in range(n_layers - 1)]
    host = [(k.pin_memory(), v.pin_memory()) for k, v in host]
    buf = [(torch.empty_like(b.k_pool, device=dev), torch.empty_like(b.v_pool, device=dev)) for _ in range(2)]
    rope = cf.rope
    q_query, q_fresh, k_fresh, v_fresh = (t.to(dev) for t in (b.q_query, b.q_fresh, b.k_fresh, b.v_fresh))
    pcf.prefetch_pool_pages(L, host[0][0], host[0][1], buf[0][0], buf[0][1])
    pcf.score(L, q_query, buf[0][0], rope, cf.importance, cf.ws_score)
    pcf.select_topk(L, cf.importance, cf.sel_idx, cf.excl, cf.row_pos)
    main, copy = torch.cuda.current_stream(), torch.cuda.Stream(device=dev)
    attn = lambda kv: pcf.fused_attention(L, q_fresh, k_fresh, v_fresh, kv[0], kv[1], cf.excl, cf.row_pos, rope,
                                          cf.out, cf.ws_attn)

    def pipelined():
        ready = [torch.cuda.Event() for _ in range(n_layers)]
        done = [torch.cuda.Event() for _ in range(n_layers)]
        with torch.cuda.stream(copy):
            pcf.prefetch_pool_pages(L, host[0][0], host[0][1], buf[0][0], buf[0][1], stream=copy)
            ready[0].record(copy)
        for l in range(n_layers):
            main.wait_event(ready[l])
            if l + 1 < n_layers:
                with torch.cuda.stream(copy):
                    if l >= 1:
                        copy.wait_event(done[l - 1])     # the buffer layer l+1 reuses is free
                    d = buf[(l + 1) & 1]
                    pcf.prefetch_pool_pages(L, host[l + 1][0], host[l + 1][1], d[0], d[1], stream=copy)
                    ready[l + 1].record(copy)
            attn(buf[l & 1])
            done[l].record(main)

    def attention_only():
        for l in range(n_layers):
            attn(buf[l & 1])

    def copies_only():
        for l in range(n_layers):
            pcf.prefetch_pool_pages(L, host[l][0], host[l][1], buf[l & 1][0], buf[l & 1][1])

    def timed(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for _ in range(reps):
            fn()
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps / n_layers

    reps = max(1, min(args.steps, 20))
    clocks = ClockSampler(local)
    clocks.start()
    ms_pipe = timed(pipelined, reps)
    clk = clocks.stop()
    ms_attn = timed(attention_only, reps)
    ms_copy = timed(copies_only, reps)
    pcf.check_device_error()
    pages = set()
    for r in b.requests:
        for sp in r.spans:
            pages.update(range(sp.phys_first_page, sp.phys_first_page + sp.n_pages))
    nbytes = 2 * len(pages) * b.hkv * PAGE * b.d * 2
    if rank == 0:
        print(json.dumps({
            "op": "layer_prefetch", "metric": "fused-attention layer time with the next layer's pool prefetched",
            "value": ms_pipe * 1e3, "unit": "us", "n_gpus": 1, "steps": reps, "warmup": 2, "ms_per_step": ms_pipe,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{args.config}: {DESCR[args.config]}", "layers": n_layers,
                       "prefetch_bytes_per_layer": nbytes, "host_pools": "pinned"},
            "attention_only_us_per_layer": ms_attn * 1e3, "copy_only_us_per_layer": ms_copy * 1e3,
            "copy_gbs": nbytes / (ms_copy / 1e3) / 1e9, "clocks": clk,
        }))


def run_op(args, pcf, b, L, cf, k_pool, dev, world, rank, local):
    """Time one selection variant alone: anchor key norms (HBM-bound: reads every cached key once)
    or the global Top-N (one block per request, launch- and latency-bound)."""
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    if args.op == "key_norms":
        # anchor extraction is offline, once per stored span: a layout that lists every span of
        # the pool once (no query, nothing recomputed)
        cfg = CONFIGS[args.config]
        pps = cfg.span_len // PAGE
        pool_req = Request(spans=[Span(i * pps, pps, i * cfg.span_len, 0) for i in range(cfg.pool_spans)],
                           n_query=0, query_pos0=cfg.pool_spans * cfg.span_len)
        L = pcf.Layout([pool_req], b.hq, b.hkv, b.d, b.n_phys_pages, cfg.pool_spans * cfg.span_len + 1,
                       device=str(dev))
    norms = torch.empty(max(1, L.total_tokens), dtype=torch.float32, device=dev)
    pcf.key_norms(L, k_pool, norms)
    offline = None
    per_call = 1
    if args.op == "key_norms":
        call = lambda: pcf.key_norms(L, k_pool, norms)
    elif args.op == "score_layers":
        from workload import layer_inputs
        qs, ks = layer_inputs(b, args.layers)
        qs, ks = [t.to(dev) for t in qs], [t.to(dev) for t in ks]
        per = torch.empty((args.layers, max(1, L.total_tokens)), dtype=torch.float32, device=dev)
        tot = torch.empty(max(1, L.total_tokens), dtype=torch.float32, device=dev)
        call = lambda: pcf.score_layers(L, qs, ks, cf.rope, per, tot, cf.ws_score)
        hw = L.host.numpy()   # per layer: rotation, LSE pass, importance pass (layout words 19, 20)
        per_call = int(args.layers * (1 + int(hw[19] > 0) + int(hw[20] > 0)) + 1)
    elif args.op == "topn_global":
        call = lambda: pcf.select_topn_global(L, norms, cf.sel_idx, cf.excl, cf.row_pos)
    else:
        call, probe_flops, offline, per_call = _anchor_probe_setup(args, pcf, b, k_pool, dev)
    for _ in range(max(3, args.warmup)):
        call()
    pcf.check_device_error()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    pcf.check_device_error()
    ms = _max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in ev), world, dev)
    peak, _, hbm, src = _peaks()
    if args.op == "anchor_probe":
        tf = world * probe_flops / (ms / 1e3) / 1e12
        metric, value, unit, hib = "anchor-prefixed query probe (fused attention) time per call", ms * 1e3, "us", False
        roof = {"bound": "tensor", "achieved": tf / world, "peak": peak, "unit": "TFLOP/s", "frac": tf / world / peak,
                "peak_source": src + " bf16 burst", "traffic": None, "algorithmic_flops_per_launch": probe_flops,
                "offline_anchor_pass_us": offline()}
    elif args.op == "score_layers":
        # one Q K^T per layer: 2*Hq*T*N*d flops per request (the implementation's two passes issue
        # twice that; both are reported)
        flops = float(args.layers * sum(2 * b.hq * r.n_query * r.n_cached * b.d for r in b.requests))
        tf = flops / (ms / 1e3) / 1e12
        metric, value, unit, hib = f"all-layer scoring ({args.layers} layers) time per call", ms * 1e3, "us", False
        roof = {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                "issued_tflops": 2 * tf, "issued_frac": 2 * tf / peak, "peak_source": src + " bf16 burst",
                "traffic": None, "algorithmic_flops_per_launch": flops}
    elif args.op == "key_norms":
        nbytes = L.total_tokens * (b.hkv * b.d * 2 + 4)     # every cached key read once, one fp32 out
        gbs = world * nbytes / (ms / 1e3) / 1e9
        metric, value, unit, hib = "anchor key norms over the span pool: key bytes read per second", gbs, "GB/s", True
        roof = {"bound": "hbm", "achieved": gbs / world, "peak": hbm, "unit": "GB/s", "frac": gbs / world / hbm,
                "peak_source": src + " copy", "traffic": None, "algorithmic_bytes_per_launch": nbytes}
    else:
        metric, value, unit, hib = "global Top-N selection time per call", ms * 1e3, "us", False
        nbytes = L.total_tokens * 4 + L.total_sel * 8 + L.total_pages * 2 + L.total_rows * 4
        gbs = nbytes / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "peak_source": src + " copy", "traffic": None, "algorithmic_bytes_per_launch": nbytes}
    if rank == 0:
        print(json.dumps({
            "op": args.op, "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "dtype": {"key_norms": "f32", "topn_global": "u32"}.get(args.op, "bf16"),
            "data": "synthetic",
            "config": {"workload": f"{args.config}: {DESCR[args.config]}", "tokens": L.total_tokens,
                       "l2": "flushed between timed calls (512 MB write)",
                       **({"layers": args.layers} if args.op == "score_layers" else {})},
            "roofline": roof, "gpu_launches": K * per_call, "clocks": clk,
        }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="batch70b", choices=list(CONFIGS))
    ap.add_argument("--pct", type=int, default=None)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="step",
                    choices=["step", "key_norms", "topn_global", "anchor_probe", "layer_prefetch",
                             "score_layers"],
                    help="step: the hot path (default); key_norms / topn_global / anchor_probe / "
                         "score_layers: one of the variants alone, on the workload's layout")
    ap.add_argument("--layers", type=int, default=4, help="score_layers: layers scored per call")
    ap.add_argument("--paged", action="store_true",
                    help="step: scoring and fused attention through pcf_score_paged / pcf_fused_attention_paged "
                         "(cached K/V read from the pool pages, keys rotated in the kernels, no per-request copy)")
    ap.add_argument("--anchor-pct", type=int, default=6,
                    help="anchor_probe: anchors per span, percent of its tokens in whole pages")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return

    world, rank, local = _dist()
    import position_independent_kv_critical_gb300 as pcf

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    b = make_batch(args.config, args.pct, shard=rank)   # each rank its own requests
    max_pos = b.max_pos + 1
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, max_pos, device=str(dev))
    rope = pcf.rope_table(b.d, b.theta, max_pos).to(dev)
    D = b.hq * b.d
    cf = pcf.CacheFusion(L, rope, row_elems=D, device=str(dev), paged=args.paged)
    g = lambda t: t.to(dev)
    k_pool, v_pool = g(b.k_pool), g(b.v_pool)
    q_query, q_fresh, k_fresh, v_fresh = g(b.q_query), g(b.q_fresh), g(b.k_fresh), g(b.v_fresh)
    if args.op == "layer_prefetch":
        run_layer_prefetch(args, pcf, b, L, cf, k_pool, dev, rank, local)
        return
    if args.op != "step":
        run_op(args, pcf, b, L, cf, k_pool, dev, world, rank, local)
        return
    hidden = hidden_rows(torch.arange(L.total_tokens, device=dev), D)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2

    def front():
        pcf.score(L, q_query, k_pool, rope, cf.importance, cf.ws_score, paged=args.paged)
        pcf.select_topk(L, cf.importance, cf.sel_idx, cf.excl, cf.row_pos)
        pcf.gather_rows(L, cf.sel_idx, hidden, cf.gathered)

    def attn():
        pcf.fused_attention(L, q_fresh, k_fresh, v_fresh, k_pool, v_pool, cf.excl, cf.row_pos, rope, cf.out,
                            cf.ws_attn, paged=args.paged)

    for _ in range(max(3, args.warmup)):
        front()
        attn()
    pcf.check_device_error()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        front()
        attn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    pcf.check_device_error()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]

    # per-call breakdown, from a separate pass: an event recorded between two calls ends the
    # overlap of the next call's first kernel with the previous call's last one, so these steps
    # are slower than the timed ones above and are used only to split the time among the calls
    Kb = min(K, 50)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Kb)]
    for i in range(Kb):
        flush.zero_()
        evb[i][0].record(stream)
        pcf.score(L, q_query, k_pool, rope, cf.importance, cf.ws_score, paged=args.paged)
        evb[i][1].record(stream)
        pcf.select_topk(L, cf.importance, cf.sel_idx, cf.excl, cf.row_pos)
        pcf.gather_rows(L, cf.sel_idx, hidden, cf.gathered)
        evb[i][2].record(stream)
        attn()
        evb[i][3].record(stream)
    torch.cuda.synchronize()
    pcf.check_device_error()
    score_ms = [e[0].elapsed_time(e[1]) for e in evb]
    topk_gather_ms = [e[1].elapsed_time(e[2]) for e in evb]
    attn_ms = [e[2].elapsed_time(e[3]) for e in evb]
    # the attention kernel alone (the dominant kernel): events recorded by the library right
    # before and after its launch, in one more pass of the same steps
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kb)]
    for i in range(Kb):
        flush.zero_()
        front()
        pcf.fused_attention(L, q_fresh, k_fresh, v_fresh, k_pool, v_pool, cf.excl, cf.row_pos, rope, cf.out,
                            cf.ws_attn, kernel_events=(evk[i][0], evk[i][1]), paged=args.paged)
    torch.cuda.synchronize()
    pcf.check_device_error()
    kernel_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evk)
    ms = _max_over_ranks(statistics.mean(step_ms), world, dev)
    tokens = sum(r.n_cached + r.n_query for r in b.requests)
    value = _job_throughput(tokens, world, ms)

    sel = cf.sel_idx[: L.total_sel].cpu().numpy()
    row_pos = cf.row_pos[: L.total_rows].cpu().numpy()
    flops = attention_flops(b, sel, row_pos, b.d, b.hq)
    a_ms = statistics.mean(attn_ms)
    peak, peak_sus, hbm, src = _peaks()
    achieved = flops / (kernel_ms / 1e3) / 1e12
    achieved_call = flops / (a_ms / 1e3) / 1e12
    score_flops = 2.0 * b.hq * b.d * sum(r.n_query * r.n_cached for r in b.requests)

    # end to end through the public API: inputs from pinned host memory, result back to the host
    hq_q = b.q_query.pin_memory()
    hq_f = [b.q_fresh.pin_memory(), b.k_fresh.pin_memory(), b.v_fresh.pin_memory()]
    out_h = torch.empty_like(cf.out, device="cpu").pin_memory()
    sel_h = torch.empty_like(cf.sel_idx, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in [hq_q] + hq_f)
    d2h = out_h.numel() * out_h.element_size() + sel_h.numel() * sel_h.element_size()
    Ke = min(K, 50)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(2):   # warm-up: the pipelined step allocates its input slots and streams once
        cf.step_from_host(hq_q, *hq_f, k_pool, v_pool, out_h, sel_h, hidden)
    cf.wait_host_results()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(Ke):
        # every step uploads its query and fresh rows and brings O and the selection back
        cf.step_from_host(hq_q, *hq_f, k_pool, v_pool, out_h, sel_h, hidden)
    cf.wait_host_results()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    pcf.check_device_error()

    hw = L.host.numpy()   # layout header: LSE items [19], importance items [20], combine items [33]
    # scoring: rotation, row LSE, importance; top-k; gather; attention: compaction scan, rotation,
    # attention, split merge
    launches_per_step = ((1 + (hw[19] > 0) + (hw[20] > 0)) if L.total_tokens else 0) + 1 + (1 if L.total_sel else 0) \
        + ((2 + (1 if L.total_tokens else 0)) if L.total_rows else 0) + (1 if hw[33] > 0 else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.config}: {DESCR[args.config]}",
                   "recompute_pct": args.pct if args.pct is not None else CONFIGS[args.config].pct,
                   "tokens_per_step": tokens, "l2": "flushed between timed steps (512 MB write)",
                   **({"attention": "paged"} if args.paged else {})},
        "roofline": {"bound": "tensor",
                     "kernel": "attn_kernel (fused attention, persistent tcgen05" +
                               (", paged: pool pages, keys rotated in shared memory)" if args.paged else ")"),
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": src + " bf16 burst", "frac_of_sustained": achieved / peak_sus if peak_sus else None,
                     "traffic": _recorded_traffic(args.config), "traffic_unit": "bytes per launch (ncu DRAM read+write)",
                     "algorithmic_flops_per_launch": flops, "ms_per_launch": kernel_ms,
                     "timing": "CUDA events recorded on the launching stream right before and after the attention "
                               "kernel's launch (pcf_fused_attention_timed), mean over a pass of the same steps",
                     "call": {"what": ("pcf_fused_attention_paged: page scan + fresh-row rotation + attention "
                                       "kernel + split merge" if args.paged else
                                       "pcf_fused_attention: compaction scan + rotation pass + attention kernel + "
                                       "split merge"), "ms": a_ms, "achieved": achieved_call,
                              "frac": achieved_call / peak,
                              "workspace_bytes": int(cf.ws_attn.numel()),
                              "score_workspace_bytes": int(cf.ws_score.numel())}},
        "breakdown_ms": {"score": statistics.mean(score_ms), "topk_gather": statistics.mean(topk_gather_ms),
                         "attention": a_ms},
        "score_tflops": score_flops / (statistics.mean(score_ms) / 1e3) / 1e12,
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": int(launches_per_step) * K,
        "clocks": clk,
        "wall_s": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle as it stands, repeated on the same requests until about 10 s of CPU work
        prep = oracle_prepare(b)
        ids, stride = _oracle_sample(b)
        t1 = time.perf_counter()
        tok = reps = 0
        dt = 0.0
        while reps < 1 or (time.perf_counter() - t1 < 10.0 and reps < 50):
            tk, sec, _, _ = oracle_step(b, prep, ids, stride)
            tok += tk
            dt += sec
            reps += 1
        line["cpu_baseline"] = {"value": tok / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                                "kind": "oracle",
                                "sample": f"{_sample_text(b, ids, stride)}, oracle step (score, top-k, gather, "
                                          f"attention; fp64 NumPy, BLAS threads = all cores) x {reps}, "
                                          f"{time.perf_counter() - t1:.1f} s of CPU time"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
