"""GB300-native query-centric cache fusion over a position-free paged KV cache.

Python binding of the C ABI in ``include/pcf.h``.  Every step of the hot path runs in the
library's sm_103a kernels; this module only marshals arguments (torch tensors -> raw pointers,
the current CUDA stream) and allocates buffers through torch.  There is no CPU fallback: without
the built library or an sm_103 device the calls raise.

Hot path for one batch at the critical layer:
  ``score``          importance of every cached token (query -> cached keys, each key rotated to its request's position at use time)
  ``select_topk``    per-span top-k tokens to recompute, exclusion bits, row positions
  ``gather_rows``    rows of the selected tokens (input of the recomputation)
  ``fused_attention`` recomputed + query rows over cached-minus-selected + fresh KV
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import PcfError  # noqa: F401

__all__ = ["Layout", "CacheFusion", "PcfError", "k_from_percent", "rope_table", "score", "select_topk",
           "gather_rows", "fused_attention", "check_device_error", "load_library", "score_noalloc",
           "select_topn_global", "key_norms", "pack_anchor_pages", "prefetch_pool_pages",
           "wait_limit_check", "score_layers"]


def load_library():
    return _lib.load()


def _p(t: Optional[torch.Tensor]):
    if t is None or t.numel() == 0:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype: torch.dtype, name: str):
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous {dtype} tensor, got {t.dtype} "
                         f"(contiguous={t.is_contiguous()})")


def k_from_percent(pct: int, span_len: int) -> int:
    return int(_lib.load().pcf_k_from_percent(int(pct), int(span_len)))


def rope_table(head_dim: int, theta: float, max_pos: int) -> torch.Tensor:
    """Host fp32 table [max_pos][head_dim/2][2] of (cos, sin)(p * theta^(-2i/d))."""
    t = torch.empty((max_pos, head_dim // 2, 2), dtype=torch.float32)
    _lib.check("pcf_rope_table_init", _lib.load().pcf_rope_table_init(
        ctypes.c_void_p(t.data_ptr()), head_dim, float(theta), max_pos))
    return t


class Layout:
    """Host + device copies of the layout blob of one batch (block table, page positions, spans,
    row offsets and work lists).  ``requests`` are objects with ``.spans`` (each with
    ``phys_first_page, n_pages, pos0, k``), ``.n_query`` and ``.query_pos0``."""

    def __init__(self, requests: Sequence, hq: int, hkv: int, d: int, n_phys_pages: int,
                 max_pos: int, device: str = "cuda"):
        lib = _lib.load()
        self._span_arrays = []
        reqs = (_lib.RequestDesc * len(requests))()
        for i, r in enumerate(requests):
            arr = (_lib.SpanDesc * max(1, len(r.spans)))()
            for j, s in enumerate(r.spans):
                arr[j] = _lib.SpanDesc(int(s.phys_first_page), int(s.n_pages), int(s.pos0), int(s.k))
            self._span_arrays.append(arr)
            reqs[i] = _lib.RequestDesc(len(r.spans), arr, int(r.n_query), int(r.query_pos0))
        # the work lists are balanced over the SMs of the device the batch runs on
        n_sms = 0
        if device != "cpu" and torch.cuda.is_available():
            n_sms = torch.cuda.get_device_properties(torch.device(device)).multi_processor_count
        dims = _lib.Dims(hq, hkv, d, n_phys_pages, max_pos, n_sms)
        n = ctypes.c_int64(0)
        _lib.check("pcf_layout_words", lib.pcf_layout_words(reqs, len(requests), ctypes.byref(dims),
                                                            ctypes.byref(n)))
        host = torch.empty(n.value, dtype=torch.int32)
        if device != "cpu" and torch.cuda.is_available():
            host = host.pin_memory()
        _lib.check("pcf_layout_build", lib.pcf_layout_build(reqs, len(requests), ctypes.byref(dims),
                                                            ctypes.c_void_p(host.data_ptr()), n.value))
        self.host = host
        self.dev = host.to(device) if device != "cpu" else host.clone()
        self.ref = _lib.LayoutRef(host.data_ptr(), self.dev.data_ptr())
        self.hq, self.hkv, self.d = hq, hkv, d
        self.requests = list(requests)

    def field(self, name: str) -> int:
        v = ctypes.c_int64(0)
        _lib.check("pcf_layout_query", _lib.load().pcf_layout_query(
            ctypes.c_void_p(self.host.data_ptr()), _lib.HEADER_FIELDS[name], ctypes.byref(v)))
        return int(v.value)

    @property
    def total_tokens(self) -> int:
        return self.field("total_tokens")

    @property
    def total_query(self) -> int:
        return self.field("total_query")

    @property
    def total_rows(self) -> int:
        return self.field("total_rows")

    @property
    def total_sel(self) -> int:
        return self.field("total_sel")

    @property
    def total_pages(self) -> int:
        return self.field("total_pages")

    def score_workspace_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _lib.check("pcf_score_workspace_bytes", _lib.load().pcf_score_workspace_bytes(
            ctypes.c_void_p(self.host.data_ptr()), ctypes.byref(v)))
        return int(v.value)

    def attention_workspace_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _lib.check("pcf_attention_workspace_bytes", _lib.load().pcf_attention_workspace_bytes(
            ctypes.c_void_p(self.host.data_ptr()), ctypes.byref(v)))
        return int(v.value)

    def score_paged_workspace_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _lib.check("pcf_score_paged_workspace_bytes", _lib.load().pcf_score_paged_workspace_bytes(
            ctypes.c_void_p(self.host.data_ptr()), ctypes.byref(v)))
        return int(v.value)

    def attention_paged_workspace_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _lib.check("pcf_attention_paged_workspace_bytes", _lib.load().pcf_attention_paged_workspace_bytes(
            ctypes.c_void_p(self.host.data_ptr()), ctypes.byref(v)))
        return int(v.value)


def score(layout: Layout, q_query, k_pool, rope, importance, ws, stream=None, paged=False):
    """``paged``: pcf_score_paged (keys read from the pool pages and rotated in the kernels; ``ws``
    sized by ``Layout.score_paged_workspace_bytes``)."""
    _need(q_query, torch.bfloat16, "q_query")
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(rope, torch.float32, "rope")
    _need(importance, torch.float32, "importance")
    fn = "pcf_score_paged" if paged else "pcf_score"
    _lib.check(fn, getattr(_lib.load(), fn)(
        ctypes.byref(layout.ref), _p(q_query), _p(k_pool), _p(rope), _p(importance), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def score_layers(layout: Layout, q_layers, k_layers, rope, importance_layers, importance_sum, ws,
                 stream=None):
    """Importance at every layer (``q_layers[l]`` over ``k_layers[l]``) into
    ``importance_layers[l]`` and their sum over the layers into ``importance_sum``."""
    if len(q_layers) != len(k_layers) or not q_layers:
        raise ValueError("q_layers and k_layers: one tensor per layer, at least one layer")
    for t in list(q_layers) + list(k_layers):
        _need(t, torch.bfloat16, "layer input")
    _need(rope, torch.float32, "rope")
    _need(importance_layers, torch.float32, "importance_layers")
    _need(importance_sum, torch.float32, "importance_sum")
    n = len(q_layers)
    qp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in q_layers])
    kp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in k_layers])
    _lib.check("pcf_score_layers", _lib.load().pcf_score_layers(
        ctypes.byref(layout.ref), n, qp, kp, _p(rope), _p(importance_layers), _p(importance_sum), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def score_noalloc(layout: Layout, q_query, k_pool, rope, importance, stream=None):
    """``score`` with the library's built-in scratch array instead of a workspace (no allocation)."""
    _need(q_query, torch.bfloat16, "q_query")
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(rope, torch.float32, "rope")
    _need(importance, torch.float32, "importance")
    _lib.check("pcf_score_noalloc", _lib.load().pcf_score_noalloc(
        ctypes.byref(layout.ref), _p(q_query), _p(k_pool), _p(rope), _p(importance), _stream(stream)))


def select_topk(layout: Layout, importance, sel_idx, excl, row_pos, stream=None):
    _need(importance, torch.float32, "importance")
    _need(sel_idx, torch.int32, "sel_idx")
    _need(excl, torch.int16, "excl")
    _need(row_pos, torch.int32, "row_pos")
    _lib.check("pcf_select_topk", _lib.load().pcf_select_topk(
        ctypes.byref(layout.ref), _p(importance), _p(sel_idx), _p(excl), _p(row_pos), _stream(stream)))


def select_topn_global(layout: Layout, importance, sel_idx, excl, row_pos, stream=None):
    """One Top-N per request over all its cached tokens (budget: the sum of its spans' k)."""
    _need(importance, torch.float32, "importance")
    _need(sel_idx, torch.int32, "sel_idx")
    _need(excl, torch.int16, "excl")
    _need(row_pos, torch.int32, "row_pos")
    _lib.check("pcf_select_topn_global", _lib.load().pcf_select_topn_global(
        ctypes.byref(layout.ref), _p(importance), _p(sel_idx), _p(excl), _p(row_pos), _stream(stream)))


def key_norms(layout: Layout, k_pool, norms, stream=None):
    """Key norm of every cached token of the layout (anchor extraction)."""
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(norms, torch.float32, "norms")
    _lib.check("pcf_key_norms", _lib.load().pcf_key_norms(
        ctypes.byref(layout.ref), _p(k_pool), _p(norms), _stream(stream)))


def pack_anchor_pages(layout: Layout, sel_idx, k_pool, v_pool, k_anchor, v_anchor, stream=None):
    """Copy the selected anchors' K/V rows into pages of their own (anchor i -> page i/16, row i%16)."""
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool"), (k_anchor, "k_anchor"), (v_anchor, "v_anchor")):
        _need(t, torch.bfloat16, n)
    _need(sel_idx, torch.int32, "sel_idx")
    _lib.check("pcf_pack_anchor_pages", _lib.load().pcf_pack_anchor_pages(
        ctypes.byref(layout.ref), _p(sel_idx), _p(k_pool), _p(v_pool), _p(k_anchor), _p(v_anchor),
        _stream(stream)))


def prefetch_pool_pages(layout: Layout, src_k, src_v, dst_k, dst_v, stream=None):
    """Queue copies of the pool pages the layout references (src -> dst, same page offsets)."""
    for t, n in ((src_k, "src_k"), (dst_k, "dst_k")):
        _need(t, torch.bfloat16, n)
    if (src_v is None) != (dst_v is None):
        raise ValueError("src_v and dst_v: both or neither")
    _lib.check("pcf_prefetch_pool_pages", _lib.load().pcf_prefetch_pool_pages(
        ctypes.byref(layout.ref), _p(src_k), _p(src_v) if src_v is not None else None, _p(dst_k),
        _p(dst_v) if dst_v is not None else None, _stream(stream)))


def gather_rows(layout: Layout, sel_idx, src, dst, stream=None):
    _need(src, torch.bfloat16, "src")
    _need(dst, torch.bfloat16, "dst")
    _lib.check("pcf_gather_rows", _lib.load().pcf_gather_rows(
        ctypes.byref(layout.ref), _p(sel_idx), _p(src), int(src.shape[-1]), _p(dst), _stream(stream)))


def fused_attention(layout: Layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl, row_pos, rope,
                    out, ws, stream=None, kernel_events=None, paged=False):
    """``paged``: the variant that reads cached K/V straight from the pool pages and rotates the
    keys in the kernel (pcf_fused_attention_paged; ``ws`` sized by
    ``Layout.attention_paged_workspace_bytes``).  ``kernel_events``: optional (start, stop)
    torch.cuda.Event pair recorded around the attention kernel alone (pcf_fused_attention_timed)."""
    for t, n in ((q_fresh, "q_fresh"), (k_fresh, "k_fresh"), (v_fresh, "v_fresh"), (k_pool, "k_pool"),
                 (v_pool, "v_pool"), (out, "out")):
        _need(t, torch.bfloat16, n)
    args = (ctypes.byref(layout.ref), _p(q_fresh), _p(k_fresh), _p(v_fresh), _p(k_pool), _p(v_pool),
            _p(excl), _p(row_pos), _p(rope), _p(out), _p(ws), ws.numel() * ws.element_size())
    if kernel_events is None:
        fn = "pcf_fused_attention_paged" if paged else "pcf_fused_attention"
        _lib.check(fn, getattr(_lib.load(), fn)(*args, _stream(stream)))
        return
    st = torch.cuda.current_stream() if stream is None else stream
    handles = []
    for ev in kernel_events:
        if not ev.cuda_event:        # torch creates its events on their first record
            ev.record(st)
        handles.append(ctypes.c_void_p(ev.cuda_event))
    _lib.check("pcf_fused_attention_timed", _lib.load().pcf_fused_attention_timed(
        *args, handles[0], handles[1], int(bool(paged)), _stream(stream)))


def wait_limit_check(limit_cycles: int, flag, stream=None):
    """Launch the bounded-wait check kernel (a wait that gives up after ``limit_cycles``); the next
    ``check_device_error`` then raises PcfError with PCF_ERR_DEVICE_TIMEOUT."""
    _need(flag, torch.int32, "flag")
    _lib.check("pcf_wait_limit_check", _lib.load().pcf_wait_limit_check(
        int(limit_cycles), _p(flag), _stream(stream)))


def check_device_error(stream=None):
    _lib.check("pcf_check_device_error", _lib.load().pcf_check_device_error(_stream(stream)))


class CacheFusion:
    """Buffers for one batch on one device plus the four calls of the hot path in order.
    ``paged=True`` runs scoring and the fused attention through pcf_score_paged and
    pcf_fused_attention_paged (no copy of the cached keys or values; workspaces that grow with the
    query and fresh rows only)."""

    def __init__(self, layout: Layout, rope_dev: torch.Tensor, row_elems: int = 0,
                 device: str = "cuda", paged: bool = False):
        L = layout
        self.layout = L
        self.rope = rope_dev
        self.paged = paged
        self.importance = torch.empty(max(1, L.total_tokens), dtype=torch.float32, device=device)
        self.sel_idx = torch.empty(max(1, L.total_sel), dtype=torch.int32, device=device)
        self.excl = torch.zeros(max(1, L.total_pages), dtype=torch.int16, device=device)
        self.row_pos = torch.empty(max(1, L.total_rows), dtype=torch.int32, device=device)
        self.out = torch.empty((max(1, L.total_rows), L.hq, L.d), dtype=torch.bfloat16, device=device)
        ws_score = L.score_paged_workspace_bytes() if paged else L.score_workspace_bytes()
        self.ws_score = torch.empty(max(16, ws_score), dtype=torch.uint8, device=device)
        ws_attn = L.attention_paged_workspace_bytes() if paged else L.attention_workspace_bytes()
        self.ws_attn = torch.empty(max(16, ws_attn), dtype=torch.uint8, device=device)
        self.gathered = (torch.empty((max(1, L.total_sel), row_elems), dtype=torch.bfloat16, device=device)
                         if row_elems else None)

    def step(self, q_query, k_pool, v_pool, q_fresh, k_fresh, v_fresh, hidden=None, stream=None):
        L = self.layout
        if getattr(self, "_ev_down", None) is not None:   # a step_from_host download may still read out
            (stream if stream is not None else torch.cuda.current_stream()).wait_event(self._ev_down)
        score(L, q_query, k_pool, self.rope, self.importance, self.ws_score, stream, paged=self.paged)
        select_topk(L, self.importance, self.sel_idx, self.excl, self.row_pos, stream)
        if hidden is not None and self.gathered is not None:
            gather_rows(L, self.sel_idx, hidden, self.gathered, stream)
        fused_attention(L, q_fresh, k_fresh, v_fresh, k_pool, v_pool, self.excl, self.row_pos,
                        self.rope, self.out, self.ws_attn, stream, paged=self.paged)
        return self.out

    def step_from_host(self, q_query_h, q_fresh_h, k_fresh_h, v_fresh_h, k_pool, v_pool, out_h, sel_h,
                       hidden=None):
        """``step`` with the per-step inputs in pinned host memory and the results (O and the
        selected token indices) copied back to pinned host buffers.

        The copies run on two streams of their own and overlap the kernels: the query rows go up
        first (scoring needs only them), the fresh Q/K/V rows while scoring runs, and the results
        come down while the next step runs.  Device input buffers alternate between two slots, so
        a step's uploads never overwrite rows the previous step's kernels may still read, and so do
        the device copies of O and the selection (slot 0 is ``out`` / ``sel_idx``), so a step's
        kernels never wait for the previous step's results to reach the host.  The host
        inputs must stay unchanged, and ``out_h`` / ``sel_h`` unread, until ``wait_host_results()``
        (or a device synchronisation) has returned."""
        L = self.layout
        lib = _lib.load()
        main = torch.cuda.current_stream()
        host_in = (q_query_h, q_fresh_h, k_fresh_h, v_fresh_h)
        if not hasattr(self, "_h2d"):
            for t in host_in + (out_h, sel_h):
                if t.is_cuda or not t.is_pinned():
                    raise ValueError("step_from_host takes pinned host tensors")
            self._h2d = torch.cuda.Stream()
            self._d2h = torch.cuda.Stream()
            self._slots = [tuple(torch.empty_like(t, device=self.out.device) for t in host_in) for _ in range(2)]
            self._out_slots = [(self.out, self.sel_idx), (torch.empty_like(self.out), torch.empty_like(self.sel_idx))]
            self._ev_q = [torch.cuda.Event() for _ in range(2)]
            self._ev_fresh = [torch.cuda.Event() for _ in range(2)]
            self._ev_used = [torch.cuda.Event() for _ in range(2)]   # slot i's last reader is done
            self._ev_down_slot = [torch.cuda.Event() for _ in range(2)]
            self._ev_down = None             # the last step's results have reached the host
            self._it = 0
        i = self._it & 1
        qq, qf, kf, vf = self._slots[i]
        out_d, sel_d = self._out_slots[i]
        n_in = [t.numel() * t.element_size() for t in host_in]
        if any(n != d.numel() * d.element_size() for n, d in zip(n_in, self._slots[i])):
            raise ValueError("step_from_host inputs changed size between steps")
        if (out_h.numel() * out_h.element_size() != self.out.numel() * self.out.element_size()
                or sel_h.numel() * sel_h.element_size() != self.sel_idx.numel() * self.sel_idx.element_size()):
            raise ValueError("step_from_host result buffers must match out and sel_idx in size")

        def copies(dst, src, nbytes, stream):
            n = len(dst)
            _lib.check("pcf_copy_async", lib.pcf_copy_async(
                n, (ctypes.c_void_p * n)(*[t.data_ptr() for t in dst]),
                (ctypes.c_void_p * n)(*[t.data_ptr() for t in src]), (ctypes.c_size_t * n)(*nbytes),
                ctypes.c_void_p(stream.cuda_stream)))

        if self._it >= 2:
            self._h2d.wait_event(self._ev_used[i])
        copies([qq], [q_query_h], n_in[:1], self._h2d)
        self._ev_q[i].record(self._h2d)
        copies([qf, kf, vf], [q_fresh_h, k_fresh_h, v_fresh_h], n_in[1:], self._h2d)
        self._ev_fresh[i].record(self._h2d)
        main.wait_event(self._ev_q[i])
        score(L, qq, k_pool, self.rope, self.importance, self.ws_score, paged=self.paged)
        if self._it >= 2:                  # this slot's results of two steps ago are on the host
            main.wait_event(self._ev_down_slot[i])
        select_topk(L, self.importance, sel_d, self.excl, self.row_pos)
        if hidden is not None and self.gathered is not None:
            gather_rows(L, sel_d, hidden, self.gathered)
        main.wait_event(self._ev_fresh[i])
        fused_attention(L, qf, kf, vf, k_pool, v_pool, self.excl, self.row_pos, self.rope, out_d,
                        self.ws_attn, paged=self.paged)
        self._ev_used[i].record(main)
        self._d2h.wait_event(self._ev_used[i])
        copies([out_h, sel_h], [out_d, sel_d],
               [out_h.numel() * out_h.element_size(), sel_h.numel() * sel_h.element_size()], self._d2h)
        self._ev_down_slot[i].record(self._d2h)
        self._ev_down = self._ev_down_slot[i]
        self._it += 1
        return out_h

    def wait_host_results(self):
        """Make the current stream wait until the last ``step_from_host`` results are on the host."""
        if getattr(self, "_ev_down", None) is not None:
            torch.cuda.current_stream().wait_event(self._ev_down)
