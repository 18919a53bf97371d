"""Helpers shared by the GPU parity tests: run the CUDA path on a workload batch and compute the
oracle's answer for the same seeded inputs (the oracle never sees a GPU value except where a test
feeds the GPU an oracle-derived input, e.g. the oracle's selection)."""
from __future__ import annotations

import numpy as np
import torch

import position_independent_kv_critical_gb300 as pcf
from oracle import method

IMP_RTOL = 1e-3          # fp32 importance: relative
OUT_ATOL, OUT_RTOL = 2e-2, 1e-2   # bf16 attention output


class GpuBatch:
    """Device copies of a workload batch plus its layout and output buffers."""

    def __init__(self, b, dev="cuda"):
        self.b = b
        self.dev = dev
        self.max_pos = max(16, b.max_pos + 1)
        self.L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, self.max_pos)
        self.rope = pcf.rope_table(b.d, b.theta, self.max_pos).to(dev)
        self.cf = pcf.CacheFusion(self.L, self.rope, row_elems=0)
        g = lambda t: t.to(dev)
        self.k_pool, self.v_pool = g(b.k_pool), g(b.v_pool)
        self.q_query = g(b.q_query)
        self.q_fresh, self.k_fresh, self.v_fresh = g(b.q_fresh), g(b.k_fresh), g(b.v_fresh)
        self.tok_base = b.token_bases()
        self.row_base = b.row_bases()
        self.sel_base = b.sel_bases()
        self.q_base = b.query_bases()
        self.page_base = [t // 16 for t in self.tok_base]

    # ---- GPU calls
    def score(self, paged=False):
        ws = self.cf.ws_score
        if paged:
            if not hasattr(self, "ws_score_paged"):
                self.ws_score_paged = torch.empty(max(16, self.L.score_paged_workspace_bytes()), dtype=torch.uint8,
                                                  device=self.dev)
            ws = self.ws_score_paged
        pcf.score(self.L, self.q_query, self.k_pool, self.rope, self.cf.importance, ws, paged=paged)
        pcf.check_device_error()
        return self.cf.importance[: self.L.total_tokens].cpu().numpy()

    def topk(self, importance_np=None):
        imp = self.cf.importance
        if importance_np is not None:
            imp = torch.as_tensor(np.asarray(importance_np, dtype=np.float32)).to(self.dev)
        pcf.select_topk(self.L, imp, self.cf.sel_idx, self.cf.excl, self.cf.row_pos)
        pcf.check_device_error()
        return (self.cf.sel_idx[: self.L.total_sel].cpu().numpy(),
                self.cf.excl[: self.L.total_pages].cpu().numpy().view(np.uint16),
                self.cf.row_pos[: self.L.total_rows].cpu().numpy())

    def attention(self, excl=None, row_pos=None, paged=False):
        """The fused attention (paged: the variant that reads the pool pages and rotates in the
        kernel, with its own, smaller workspace)."""
        ex = self.cf.excl if excl is None else torch.as_tensor(
            np.asarray(excl, dtype=np.uint16).view(np.int16)).to(self.dev)
        rp = self.cf.row_pos if row_pos is None else torch.as_tensor(
            np.asarray(row_pos, dtype=np.int32)).to(self.dev)
        ws = self.cf.ws_attn
        if paged:
            if not hasattr(self, "ws_paged"):
                self.ws_paged = torch.empty(max(16, self.L.attention_paged_workspace_bytes()), dtype=torch.uint8,
                                            device=self.dev)
            ws = self.ws_paged
        pcf.fused_attention(self.L, self.q_fresh, self.k_fresh, self.v_fresh, self.k_pool, self.v_pool,
                            ex, rp, self.rope, self.cf.out, ws, paged=paged)
        pcf.check_device_error()
        return self.cf.out[: self.L.total_rows].float().cpu().numpy()

    # ---- oracle side (fp64, CPU)
    def oracle_request(self, i):
        b = self.b
        r = b.requests[i]
        if not hasattr(self, "_pool64"):    # exact fp64 copies of the bf16 pools, made once
            self._pool64 = (b.k_pool.double().numpy(), b.v_pool.double().numpy())
        K, V, kpos = method.request_cached(r.spans, *self._pool64)
        return r, K, V, kpos

    def oracle_score(self, i):
        r, K, V, kpos = self.oracle_request(i)
        q = self.b.q_query[self.q_base[i]: self.q_base[i] + r.n_query].double().numpy()
        return method.score_request(q, r.query_pos0 + np.arange(r.n_query), K, kpos, self.b.theta)

    def oracle_select(self, i, imp32):
        r = self.b.requests[i]
        return method.select_topk_request(imp32, [s.n_pages * 16 for s in r.spans], [s.k for s in r.spans])

    def oracle_attention(self, i, sel, rows=None):
        r, K, V, kpos = self.oracle_request(i)
        rb = self.row_base[i]
        sl = slice(rb, rb + r.n_rows)
        row_pos = method.row_positions(sel, kpos, r.n_query, r.query_pos0)
        return method.fused_attention_request(self.b.q_fresh[sl].double().numpy(),
                                              self.b.k_fresh[sl].double().numpy(),
                                              self.b.v_fresh[sl].double().numpy(), row_pos, K, V,
                                              kpos, sel, self.b.theta, rows=rows), row_pos

    def selection_inputs(self, sels):
        """Device-format exclusion masks and row positions for per-request selections."""
        excl = np.zeros(self.L.total_pages, dtype=np.uint16)
        row_pos = np.zeros(self.L.total_rows, dtype=np.int32)
        for i, r in enumerate(self.b.requests):
            kpos = (np.concatenate([s.pos0 + np.arange(s.n_pages * 16) for s in r.spans])
                    if r.spans else np.zeros(0, dtype=np.int64))
            npg = sum(s.n_pages for s in r.spans)
            excl[self.page_base[i]: self.page_base[i] + npg] = method.exclusion_masks(sels[i], npg)
            row_pos[self.row_base[i]: self.row_base[i] + r.n_rows] = method.row_positions(
                sels[i], kpos, r.n_query, r.query_pos0)
        return excl, row_pos


def assert_close_out(got, exp, what=""):
    err = np.abs(got - exp)
    lim = OUT_ATOL + OUT_RTOL * np.abs(exp)
    bad = err > lim
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs outside 2e-2 abs + 1e-2 rel; "
                           f"max err {err.max():.3e}")


def assert_close_imp(got, exp, what=""):
    err = np.abs(got - exp)
    lim = IMP_RTOL * np.abs(exp) + 1e-7
    bad = err > lim
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} importances outside 1e-3 rel; "
                           f"max rel err {(err / np.maximum(np.abs(exp), 1e-30)).max():.3e}")
