"""The allocation-free scoring entry point (pcf_score_noalloc), called through the C ABI.

Some callers cannot allocate device memory on the scoring path (an engine whose pool already owns
the device memory, fixed-budget real-time deployments, plugin hosts without access to an
allocator).  pcf_score_noalloc serves them from a scratch array built into the library.  These
tests check that it returns what pcf_score returns, on two calls in a row (the array keeps the
previous call's contents, so the second call must not depend on them), and that it refuses a
batch that needs more scratch than the array holds.  This file is collected last on purpose.
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


def _setup(name):
    b = make_batch(name)
    max_pos = b.max_pos + 1
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, max_pos)
    rope = pcf.rope_table(b.d, b.theta, max_pos).cuda()
    return b, L, rope, b.q_query.cuda(), b.k_pool.cuda()


def _noalloc(lib, L, q, k, rope, imp):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pcf_score_noalloc(ctypes.byref(L.ref), ctypes.c_void_p(q.data_ptr()),
                                 ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(rope.data_ptr()),
                                 ctypes.c_void_p(imp.data_ptr()), stream)


def test_noalloc_matches_score_on_two_calls_in_a_row():
    lib = _lib.load()
    for name in ("llama8b_layer", "tiny"):
        b, L, rope, q, k = _setup(name)
        assert L.score_workspace_bytes() <= (16 << 20)
        ref = torch.empty(L.total_tokens, dtype=torch.float32, device="cuda")
        ws = torch.empty(L.score_workspace_bytes(), dtype=torch.uint8, device="cuda")
        pcf.score(L, q, k, rope, ref, ws)
        got = torch.full((L.total_tokens,), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, L, q, k, rope, got) == 0
        pcf.check_device_error()
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.all(np.abs(g - r) <= IMP_RTOL * np.abs(r) + 1e-7), name


def test_noalloc_rejects_a_batch_beyond_its_array():
    lib = _lib.load()
    b = make_batch("concurrent_reuse")
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, b.max_pos + 1)
    assert L.score_workspace_bytes() > (16 << 20)
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, L, t, t, t, t) == -5     # PCF_ERR_WORKSPACE_TOO_SMALL, nothing launched
    pcf.check_device_error()
