"""The allocation-free scoring entry point (pcf_score_noalloc), called through the C ABI.

Some callers cannot allocate device memory on the scoring path: an engine whose memory pool has
already reserved the device, a real-time deployment with a fixed memory budget, or a plugin host
whose allocator the library cannot reach.  pcf_score_noalloc serves them from a scratch array
built into the library.  These tests check that it returns what pcf_score returns on two calls
in a row with the same batch (the array keeps the previous call's counters and partial sums at
the very same offsets, so the second call shows whether anything depends on that state), through
the C ABI on the current stream and through the Python binding on a side stream, and that it
refuses a batch that needs more scratch than the array holds.  This file is collected last on
purpose: the scratch array then starts dirty from the earlier tests' calls as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import position_independent_kv_critical_gb300 as pcf
from position_independent_kv_critical_gb300 import _lib
from workload import make_batch

pytestmark = pytest.mark.gpu

IMP_RTOL = 1e-3
ARRAY_BYTES = 16 << 20


def _setup(name):
    b = make_batch(name)
    max_pos = b.max_pos + 1
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, max_pos)
    rope = pcf.rope_table(b.d, b.theta, max_pos).cuda()
    return b, L, rope, b.q_query.cuda(), b.k_pool.cuda()


def _noalloc(lib, L, q, k, rope, imp, stream=None):
    st = torch.cuda.current_stream() if stream is None else stream
    return lib.pcf_score_noalloc(ctypes.byref(L.ref), ctypes.c_void_p(q.data_ptr()),
                                 ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(rope.data_ptr()),
                                 ctypes.c_void_p(imp.data_ptr()), ctypes.c_void_p(st.cuda_stream))


def _close(got, ref):
    g, r = got.cpu().numpy(), ref.cpu().numpy()
    return bool(np.all(np.isfinite(g)) and np.all(np.abs(g - r) <= IMP_RTOL * np.abs(r) + 1e-7))


@pytest.mark.parametrize("name", ["llama8b_layer", "tiny"])
def test_noalloc_matches_score_on_two_calls_in_a_row(name):
    lib = _lib.load()
    b, L, rope, q, k = _setup(name)
    assert L.score_workspace_bytes() <= ARRAY_BYTES
    ref = torch.empty(L.total_tokens, dtype=torch.float32, device="cuda")
    ws = torch.empty(L.score_workspace_bytes(), dtype=torch.uint8, device="cuda")
    pcf.score(L, q, k, rope, ref, ws)
    for call in range(2):
        got = torch.full((L.total_tokens,), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, L, q, k, rope, got) == 0
        pcf.check_device_error()
        assert _close(got, ref), f"{name}, call {call + 1}"


def test_noalloc_binding_on_a_side_stream_twice():
    b, L, rope, q, k = _setup("llama8b_layer")
    ref = torch.empty(L.total_tokens, dtype=torch.float32, device="cuda")
    ws = torch.empty(L.score_workspace_bytes(), dtype=torch.uint8, device="cuda")
    pcf.score(L, q, k, rope, ref, ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    for call in range(2):
        got = torch.full((L.total_tokens,), float("nan"), dtype=torch.float32, device="cuda")
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            pcf.score_noalloc(L, q, k, rope, got)
        torch.cuda.current_stream().wait_stream(side)
        pcf.check_device_error(side)
        assert _close(got, ref), f"side stream, call {call + 1}"


def test_noalloc_rejects_a_batch_beyond_its_array():
    lib = _lib.load()
    b = make_batch("concurrent_reuse")
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, b.max_pos + 1)
    assert L.score_workspace_bytes() > ARRAY_BYTES
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, L, t, t, t, t) == -5     # PCF_ERR_WORKSPACE_TOO_SMALL, nothing launched
    pcf.check_device_error()
