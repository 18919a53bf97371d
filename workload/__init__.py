"""Seeded synthetic workloads for query-centric cache fusion over a position-free KV cache.

This module only *generates inputs*: span layouts, logical positions and bf16 tensors drawn from
seeded CPU generators.  It holds none of the method's arithmetic (no rotation, no softmax, no
selection), so both the fp64 oracle (``oracle/``) and the CUDA path read identical bits from it.

Five named workloads are defined (sizes from the build's benchmark definition):

* ``tiny``            1 request, 8 q / 2 kv heads, d=64, 4 spans x 128 tokens at offsets
                      0/128/256/384, 32 query tokens, theta=1e4, recompute 15 % per span.
* ``llama8b_layer``   32 q / 8 kv heads, d=128, 1 request of 8 spans x 512 tokens at a random
                      base offset, 64 query tokens, theta=5e5, recompute 15 %.
* ``concurrent_reuse`` 32 requests over a shared pool of 64 spans x 1024 tokens; each request
                      draws 10 spans by Zipf(1.1) without replacement at a random base offset,
                      so one physical page serves several logical offsets; 64 query tokens, 15 %.
* ``long_context``    1 request, 64 spans x 512 = 32768 cached tokens, 128 query tokens;
                      recompute sweep 5/10/15/20/30 %.
* ``batch70b``        64 q / 8 kv heads, 64 requests x 16 spans x 1024 tokens from a pool of
                      256 spans (Zipf(1.0)), 128 query tokens, recompute 10 %.

Readings of what the source pages leave open:
* a request's spans are laid contiguously in draw order from a base offset b ~ U{0..4095};
* Zipf draws are without replacement (a document appears once per prompt), rank probability
  proportional to r^-a over the pool;
* the query tokens follow the last span immediately (query_pos0 = end of the last span);
* fresh Q/K/V of recomputed rows are independent N(0,1) draws; the query rows of q_fresh are the
  scoring query itself (the same tokens at the same layer);
* theta for the three large workloads is 5e5 (stated only for the Llama-3-8B-shaped layer).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

PAGE = 16  # tokens per KV page


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    index: int            # 1-based position in the benchmark definition; master seed = index*1000+17
    n_reqs: int
    hq: int
    hkv: int
    d: int
    theta: float
    span_len: int
    pool_spans: int
    spans_per_req: int
    n_query: int
    pct: int
    zipf: Optional[float] = None          # None: every request takes the whole pool (permuted)
    fixed_offsets: Optional[Sequence[int]] = None  # explicit span positions (tiny workload)
    pct_sweep: Optional[Sequence[int]] = None

    @property
    def seed(self) -> int:
        return self.index * 1000 + 17

    def shard_seed(self, shard: int) -> int:
        """Master seed of shard ``shard`` of the workload (one per rank under weak scaling): shard 0
        is the workload itself; the others draw different requests of the same shape."""
        return self.seed + 7919 * int(shard)


CONFIGS = {
    "tiny": WorkloadConfig("tiny", 1, n_reqs=1, hq=8, hkv=2, d=64, theta=1e4, span_len=128,
                           pool_spans=4, spans_per_req=4, n_query=32, pct=15,
                           fixed_offsets=(0, 128, 256, 384)),
    "llama8b_layer": WorkloadConfig("llama8b_layer", 2, n_reqs=1, hq=32, hkv=8, d=128, theta=5e5,
                                    span_len=512, pool_spans=8, spans_per_req=8, n_query=64,
                                    pct=15),
    "concurrent_reuse": WorkloadConfig("concurrent_reuse", 3, n_reqs=32, hq=32, hkv=8, d=128,
                                       theta=5e5, span_len=1024, pool_spans=64, spans_per_req=10,
                                       n_query=64, pct=15, zipf=1.1),
    "long_context": WorkloadConfig("long_context", 4, n_reqs=1, hq=32, hkv=8, d=128, theta=5e5,
                                   span_len=512, pool_spans=64, spans_per_req=64, n_query=128,
                                   pct=15, pct_sweep=(5, 10, 15, 20, 30)),
    "batch70b": WorkloadConfig("batch70b", 5, n_reqs=64, hq=64, hkv=8, d=128, theta=5e5,
                               span_len=1024, pool_spans=256, spans_per_req=16, n_query=128,
                               pct=10, zipf=1.0),
}


@dataclasses.dataclass
class Span:
    phys_first_page: int   # first physical page of the span in the pool (span pages are consecutive)
    n_pages: int
    pos0: int              # logical position of the span's first token in this request
    k: int                 # tokens of this span to recompute


@dataclasses.dataclass
class Request:
    spans: List[Span]
    n_query: int
    query_pos0: int

    @property
    def n_cached(self) -> int:
        return sum(s.n_pages for s in self.spans) * PAGE

    @property
    def n_sel(self) -> int:
        return sum(s.k for s in self.spans)

    @property
    def n_rows(self) -> int:
        return self.n_sel + self.n_query


@dataclasses.dataclass
class Batch:
    """Host description of one batch plus its seeded tensors (CPU, bf16)."""
    cfg_name: str
    hq: int
    hkv: int
    d: int
    theta: float
    n_phys_pages: int
    requests: List[Request]
    k_pool: torch.Tensor   # [P_phys][Hkv][16][d] bf16, keys stored unrotated
    v_pool: torch.Tensor   # [P_phys][Hkv][16][d] bf16
    q_query: torch.Tensor  # [sum T][Hq][d] bf16, unrotated
    q_fresh: torch.Tensor  # [sum rows][Hq][d] bf16 (rows: selected tokens, then query tokens)
    k_fresh: torch.Tensor  # [sum rows][Hkv][d] bf16
    v_fresh: torch.Tensor  # [sum rows][Hkv][d] bf16
    seed: int

    @property
    def max_pos(self) -> int:
        return max(r.query_pos0 + r.n_query for r in self.requests)

    def token_bases(self) -> List[int]:
        out, acc = [], 0
        for r in self.requests:
            out.append(acc)
            acc += r.n_cached
        return out

    def query_bases(self) -> List[int]:
        out, acc = [], 0
        for r in self.requests:
            out.append(acc)
            acc += r.n_query
        return out

    def row_bases(self) -> List[int]:
        out, acc = [], 0
        for r in self.requests:
            out.append(acc)
            acc += r.n_rows
        return out

    def sel_bases(self) -> List[int]:
        out, acc = [], 0
        for r in self.requests:
            out.append(acc)
            acc += r.n_sel
        return out

    @property
    def total_tokens(self) -> int:
        return sum(r.n_cached for r in self.requests)

    @property
    def total_query(self) -> int:
        return sum(r.n_query for r in self.requests)

    @property
    def total_rows(self) -> int:
        return sum(r.n_rows for r in self.requests)

    @property
    def total_sel(self) -> int:
        return sum(r.n_sel for r in self.requests)


def recompute_count(pct: int, length: int) -> int:
    """Tokens to recompute in a span of ``length`` at ``pct`` percent: ceil(pct*length/100) in
    integers.  Used here only to size the fresh-row tensors; the oracle and the C library each
    compute it on their own."""
    return -((-pct * length) // 100)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, seed: int) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(seed), dtype=torch.float32).to(torch.bfloat16)


def _zipf_draw(rng: np.random.Generator, n_pool: int, n_draw: int, a: float) -> List[int]:
    """n_draw distinct pool indices; rank r (1-based) has probability proportional to r^-a."""
    w = np.arange(1, n_pool + 1, dtype=np.float64) ** (-a)
    p = w / w.sum()
    return [int(x) for x in rng.choice(n_pool, size=n_draw, replace=False, p=p)]


def make_layout(cfg: WorkloadConfig, pct: Optional[int] = None, shard: int = 0) -> List[Request]:
    """Span placement for every request of ``cfg`` (seeded, deterministic; ``shard`` > 0 draws
    another set of requests with the same sizes)."""
    pct = cfg.pct if pct is None else pct
    rng = np.random.default_rng(cfg.shard_seed(shard))
    pages_per_span = cfg.span_len // PAGE
    reqs: List[Request] = []
    for _ in range(cfg.n_reqs):
        if cfg.zipf is None:
            order = list(range(cfg.pool_spans))
            if cfg.fixed_offsets is None:
                order = [int(x) for x in rng.permutation(cfg.pool_spans)][: cfg.spans_per_req]
            else:
                order = order[: cfg.spans_per_req]
        else:
            order = _zipf_draw(rng, cfg.pool_spans, cfg.spans_per_req, cfg.zipf)
        if cfg.fixed_offsets is not None:
            offsets = list(cfg.fixed_offsets)
        else:
            base = int(rng.integers(0, 4096))
            offsets = [base + i * cfg.span_len for i in range(len(order))]
        spans = [Span(phys_first_page=sid * pages_per_span, n_pages=pages_per_span, pos0=off,
                      k=recompute_count(pct, cfg.span_len))
                 for sid, off in zip(order, offsets)]
        qpos0 = spans[-1].pos0 + spans[-1].n_pages * PAGE
        reqs.append(Request(spans=spans, n_query=cfg.n_query, query_pos0=qpos0))
    return reqs


def make_batch_from_requests(name: str, requests: List[Request], hq: int, hkv: int, d: int,
                             theta: float, n_phys_pages: int, seed: int) -> Batch:
    """Draw every tensor for a given request list.  Sub-seeds: pool K = seed+1, pool V = seed+2,
    query Q = seed+3, fresh Q = seed+4, fresh K = seed+5, fresh V = seed+6."""
    total_q = sum(r.n_query for r in requests)
    total_rows = sum(r.n_rows for r in requests)
    k_pool = _randn_bf16((n_phys_pages, hkv, PAGE, d), seed + 1)
    v_pool = _randn_bf16((n_phys_pages, hkv, PAGE, d), seed + 2)
    q_query = _randn_bf16((total_q, hq, d), seed + 3)
    q_fresh = _randn_bf16((total_rows, hq, d), seed + 4)
    k_fresh = _randn_bf16((total_rows, hkv, d), seed + 5)
    v_fresh = _randn_bf16((total_rows, hkv, d), seed + 6)
    # the query rows of q_fresh are the scoring query itself
    qb, rb = 0, 0
    for r in requests:
        q_fresh[rb + r.n_sel: rb + r.n_rows] = q_query[qb: qb + r.n_query]
        qb += r.n_query
        rb += r.n_rows
    return Batch(cfg_name=name, hq=hq, hkv=hkv, d=d, theta=theta, n_phys_pages=n_phys_pages,
                 requests=requests, k_pool=k_pool, v_pool=v_pool, q_query=q_query,
                 q_fresh=q_fresh, k_fresh=k_fresh, v_fresh=v_fresh, seed=seed)


def make_batch(cfg_name: str, pct: Optional[int] = None, shard: int = 0) -> Batch:
    """The workload's batch; ``shard`` r > 0 gives rank r of a weak-scaling run its own requests
    and tensors (same shapes, token counts and statistics, other draws)."""
    cfg = CONFIGS[cfg_name]
    reqs = make_layout(cfg, pct, shard)
    n_phys = cfg.pool_spans * (cfg.span_len // PAGE)
    return make_batch_from_requests(cfg.name, reqs, cfg.hq, cfg.hkv, cfg.d, cfg.theta, n_phys,
                                    cfg.shard_seed(shard))


def layer_inputs(b: Batch, n_layers: int):
    """Per-layer scoring inputs for all-layer importance: layer 0 is the batch's own query and key
    pool, layer l >= 1 draws both anew (query seed + 1000 + 2l, keys seed + 1001 + 2l), same shapes
    and positions.  Returns (query list, key-pool list), CPU bf16."""
    qs, ks = [b.q_query], [b.k_pool]
    for l in range(1, n_layers):
        qs.append(_randn_bf16(tuple(b.q_query.shape), b.seed + 1000 + 2 * l))
        ks.append(_randn_bf16(tuple(b.k_pool.shape), b.seed + 1001 + 2 * l))
    return qs, ks


def hidden_rows(tok: torch.Tensor, row_elems: int) -> torch.Tensor:
    """Deterministic stand-in for per-token hidden states, evaluable for any token subset on any
    device: value(tok, col) = ((tok*131 + col*7) mod 512 - 256) / 64, exact in bf16."""
    col = torch.arange(row_elems, device=tok.device, dtype=torch.int64)
    v = (tok.to(torch.int64)[:, None] * 131 + col[None, :] * 7) % 512 - 256
    return (v.to(torch.float32) / 64.0).to(torch.bfloat16)


def small_custom_batch(spans, n_query, query_pos0=None, hq=4, hkv=2, d=64, theta=1e4,
                       seed=4242, n_phys_pages=None, extra_requests=()) -> Batch:
    """A hand-placed batch for edge cases: ``spans`` is a list of (phys_first_page, n_pages, pos0, k)
    for request 0; ``extra_requests`` holds (spans, n_query, query_pos0) tuples for more requests."""
    def mk(sp, nq, qp):
        ss = [Span(*s) for s in sp]
        if qp is None:
            qp = (ss[-1].pos0 + ss[-1].n_pages * PAGE) if ss else 0
        return Request(spans=ss, n_query=nq, query_pos0=qp)

    reqs = [mk(spans, n_query, query_pos0)] + [mk(*e) for e in extra_requests]
    if n_phys_pages is None:
        n_phys_pages = max([s.phys_first_page + s.n_pages for r in reqs for s in r.spans] + [1])
    return make_batch_from_requests("custom", reqs, hq, hkv, d, theta, n_phys_pages, seed)
