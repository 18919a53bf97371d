"""ctypes view of the C ABI declared in include/pcf.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

c_int32 = ctypes.c_int32
c_int64 = ctypes.c_int64
c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t

PCF_OK = 0
STATUS = {
    0: "PCF_OK", -1: "PCF_ERR_INVALID_ARG", -2: "PCF_ERR_UNSUPPORTED", -3: "PCF_ERR_CUDA",
    -4: "PCF_ERR_DEVICE_TIMEOUT", -5: "PCF_ERR_WORKSPACE_TOO_SMALL", -6: "PCF_ERR_DEVICE_BOUNDS",
    -7: "PCF_ERR_NO_DEVICE", -8: "PCF_ERR_DEVICE_RANGE",
}
HEADER_FIELDS = {
    "words": 1, "n_reqs": 2, "hq": 3, "hkv": 4, "d": 5, "n_phys_pages": 6, "max_pos": 7,
    "total_tokens": 8, "total_query": 9, "total_rows": 10, "total_sel": 11, "total_pages": 12,
    "n_spans": 13,
}

# every symbol include/pcf.h declares
EXPORTS = (
    "pcf_status_string", "pcf_k_from_percent", "pcf_rope_table_init", "pcf_layout_words",
    "pcf_layout_build", "pcf_layout_query", "pcf_score_workspace_bytes", "pcf_score",
    "pcf_select_topk", "pcf_gather_rows", "pcf_attention_workspace_bytes", "pcf_fused_attention",
    "pcf_check_device_error", "pcf_score_noalloc", "pcf_copy_async", "pcf_select_topn_global",
    "pcf_key_norms", "pcf_pack_anchor_pages", "pcf_prefetch_pool_pages", "pcf_fused_attention_timed",
    "pcf_wait_limit_check", "pcf_score_layers", "pcf_fused_attention_paged",
    "pcf_attention_paged_workspace_bytes", "pcf_score_paged", "pcf_score_paged_workspace_bytes",
)


class SpanDesc(ctypes.Structure):
    _fields_ = [("phys_first_page", c_int32), ("n_pages", c_int32), ("pos0", c_int32), ("k", c_int32)]


class RequestDesc(ctypes.Structure):
    _fields_ = [("n_spans", c_int32), ("spans", ctypes.POINTER(SpanDesc)), ("n_query", c_int32),
                ("query_pos0", c_int32)]


class Dims(ctypes.Structure):
    _fields_ = [("n_q_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32),
                ("n_phys_pages", c_int32), ("max_pos", c_int32), ("n_sms", c_int32)]


class LayoutRef(ctypes.Structure):
    _fields_ = [("host", c_void_p), ("dev", c_void_p)]


class PcfError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({text})")
        self.status = status


_lock = threading.Lock()
_lib = None


def _declare(lib):
    P = ctypes.POINTER
    lib.pcf_status_string.restype = ctypes.c_char_p
    lib.pcf_status_string.argtypes = [c_int32]
    lib.pcf_k_from_percent.restype = c_int32
    lib.pcf_k_from_percent.argtypes = [c_int32, c_int32]
    lib.pcf_rope_table_init.restype = c_int32
    lib.pcf_rope_table_init.argtypes = [c_void_p, c_int32, ctypes.c_double, c_int32]
    lib.pcf_layout_words.restype = c_int32
    lib.pcf_layout_words.argtypes = [P(RequestDesc), c_int32, P(Dims), P(c_int64)]
    lib.pcf_layout_build.restype = c_int32
    lib.pcf_layout_build.argtypes = [P(RequestDesc), c_int32, P(Dims), c_void_p, c_int64]
    lib.pcf_layout_query.restype = c_int32
    lib.pcf_layout_query.argtypes = [c_void_p, c_int32, P(c_int64)]
    for fn in ("pcf_score_workspace_bytes", "pcf_attention_workspace_bytes", "pcf_attention_paged_workspace_bytes",
               "pcf_score_paged_workspace_bytes"):
        getattr(lib, fn).restype = c_int32
        getattr(lib, fn).argtypes = [c_void_p, P(c_size_t)]
    lib.pcf_score.restype = c_int32
    lib.pcf_score.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.pcf_score_paged.restype = c_int32
    lib.pcf_score_paged.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.pcf_score_layers.restype = c_int32
    lib.pcf_score_layers.argtypes = [P(LayoutRef), c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_size_t, c_void_p]
    lib.pcf_select_topk.restype = c_int32
    lib.pcf_select_topk.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.pcf_select_topn_global.restype = c_int32
    lib.pcf_select_topn_global.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.pcf_key_norms.restype = c_int32
    lib.pcf_key_norms.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p]
    lib.pcf_pack_anchor_pages.restype = c_int32
    lib.pcf_pack_anchor_pages.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.pcf_prefetch_pool_pages.restype = c_int32
    lib.pcf_prefetch_pool_pages.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.pcf_gather_rows.restype = c_int32
    lib.pcf_gather_rows.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_int32, c_void_p, c_void_p]
    lib.pcf_fused_attention.restype = c_int32
    lib.pcf_fused_attention.argtypes = [P(LayoutRef)] + [c_void_p] * 10 + [c_size_t, c_void_p]
    lib.pcf_fused_attention_timed.restype = c_int32
    lib.pcf_fused_attention_paged.restype = c_int32
    lib.pcf_fused_attention_paged.argtypes = [P(LayoutRef)] + [c_void_p] * 10 + [c_size_t, c_void_p]
    lib.pcf_fused_attention_timed.argtypes = [P(LayoutRef)] + [c_void_p] * 10 + [c_size_t] + [c_void_p] * 2 + [c_int32, c_void_p]
    lib.pcf_score_noalloc.restype = c_int32
    lib.pcf_score_noalloc.argtypes = [P(LayoutRef), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.pcf_check_device_error.restype = c_int32
    lib.pcf_check_device_error.argtypes = [c_void_p]
    lib.pcf_wait_limit_check.restype = c_int32
    lib.pcf_wait_limit_check.argtypes = [c_int64, c_void_p, c_void_p]
    lib.pcf_copy_async.restype = c_int32
    lib.pcf_copy_async.argtypes = [c_int32, c_void_p, c_void_p, c_void_p, c_void_p]


def load(build_if_missing: bool = True):
    """Load (building first if needed) the in-tree library.  Raises if it cannot be built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.library_path()
            if build_if_missing:
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library missing: {path} (run __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            _declare(lib)
            _lib = lib
    return _lib


def check(fn: str, status: int) -> None:
    if status != PCF_OK:
        text = load().pcf_status_string(status).decode()
        raise PcfError(fn, status, text)
