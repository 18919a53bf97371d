"""Host-side tests of the C ABI (CPU only, no device compute): exports, layout build and
validation, RoPE table, recompute counts."""
import ctypes
import math
import os
import re

import numpy as np
import pytest
import torch

import position_independent_kv_critical_gb300 as pcf
from position_independent_kv_critical_gb300 import _lib
from workload import CONFIGS, PAGE, make_layout, small_custom_batch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")

# word map of the blob (mirrors the library's internal layout format; checked against totals)
L_OFF_REQ, L_OFF_SPAN, L_OFF_BLOCK, L_OFF_PAGEPOS = 24, 25, 26, 27
L_OFF_ATTN, L_OFF_LSE, L_OFF_IMP, L_OFF_QPOS = 28, 29, 30, 31
L_N_ATTN, L_N_LSE, L_N_IMP = 18, 19, 20
L_OFF_COMB, L_N_COMB, L_OFF_PAIR, L_N_PAIRS = 32, 33, 35, 36


def test_library_exports_every_declared_symbol(lib):
    with open(os.path.join(ROOT, "include", "pcf.h")) as fh:
        text = fh.read()
    declared = set(re.findall(r"^\s*(?:pcf_status|const char\*|int32_t)\s+(pcf_\w+)\s*\(", text, re.M))
    assert declared == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_copy_async_rejects_bad_arguments_before_touching_a_device(lib):
    PCF_OK, PCF_ERR_INVALID_ARG = 0, -1
    assert lib.pcf_copy_async(-1, None, None, None, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_copy_async(2, None, None, None, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_copy_async(0, None, None, None, None) == PCF_OK


def test_status_strings(lib):
    for code in range(-7, 1):
        s = lib.pcf_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.pcf_status_string(-99).decode() == "unknown status"


def test_k_from_percent_matches_golden(lib):
    with open(os.path.join(GOLDEN, "recompute_counts.txt")) as fh:
        rows = [ln.split("#")[0].split() for ln in fh if ln.split("#")[0].strip()]
    for pct, L, k in rows:
        assert lib.pcf_k_from_percent(int(pct), int(L)) == int(k)
    assert lib.pcf_k_from_percent(-1, 10) == -1


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 5e5)])
def test_rope_table_within_one_ulp_of_fp64(d, theta):
    max_pos = 4096
    t = pcf.rope_table(d, theta, max_pos).numpy()
    inv = theta ** (-2.0 * np.arange(d // 2) / d)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    for k, f in ((0, np.cos), (1, np.sin)):
        ref = f(ang)
        got = t[:, :, k].astype(np.float64)
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(got - ref) <= ulp)


def test_rope_table_rejects_bad_args(lib):
    buf = torch.empty(16 * 32 * 2, dtype=torch.float32)
    p = ctypes.c_void_p(buf.data_ptr())
    assert lib.pcf_rope_table_init(None, 64, 1e4, 16) == -1
    assert lib.pcf_rope_table_init(p, 96, 1e4, 16) == -2
    assert lib.pcf_rope_table_init(p, 64, 0.0, 16) == -1
    assert lib.pcf_rope_table_init(p, 64, 1e4, 8) == -1


def _blob(layout):
    return layout.host.numpy()


@pytest.mark.parametrize("name,grouped", [("batch70b", True), ("concurrent_reuse", True),
                                          ("long_context", False), ("llama8b_layer", False)])
def test_attention_items_grouped_by_unit_when_many(name, grouped):
    """With many attention items per SM the work list keeps each (request, kv head) unit's items
    in one run, so that the CTAs running at one time share a few units' keys in L2; with few
    (small batches) the list stays longest-first, which interleaves the units."""
    cfg = CONFIGS[name]
    reqs = make_layout(cfg)
    n_phys = cfg.pool_spans * cfg.span_len // PAGE
    max_pos = max(r.query_pos0 + r.n_query for r in reqs)
    L = pcf.Layout(reqs, cfg.hq, cfg.hkv, cfg.d, n_phys, max_pos, device="cpu")
    B = _blob(L)
    items = B[B[L_OFF_ATTN]: B[L_OFF_ATTN] + 4 * B[L_N_ATTN]].reshape(-1, 4)
    assert (len(items) >= 8 * int(B[37])) == grouped
    units = [(int(r), int(h)) for r, h, _, _ in items]
    runs = sum(1 for i in range(len(units)) if i == 0 or units[i] != units[i - 1])
    assert (runs == len(set(units))) == grouped


@pytest.mark.parametrize("name", list(CONFIGS))
def test_layout_totals_and_block_table(name):
    cfg = CONFIGS[name]
    reqs = make_layout(cfg)
    n_phys = cfg.pool_spans * cfg.span_len // PAGE
    max_pos = max(r.query_pos0 + r.n_query for r in reqs)
    L = pcf.Layout(reqs, cfg.hq, cfg.hkv, cfg.d, n_phys, max_pos, device="cpu")
    assert L.total_tokens == sum(r.n_cached for r in reqs)
    assert L.total_query == sum(r.n_query for r in reqs)
    assert L.total_sel == sum(r.n_sel for r in reqs)
    assert L.total_rows == sum(r.n_rows for r in reqs)
    assert L.total_pages * PAGE == L.total_tokens
    B = _blob(L)
    blk = B[B[L_OFF_BLOCK]: B[L_OFF_BLOCK] + L.total_pages]
    ppos = B[B[L_OFF_PAGEPOS]: B[L_OFF_PAGEPOS] + L.total_pages]
    exp_blk = [s.phys_first_page + i for r in reqs for s in r.spans for i in range(s.n_pages)]
    exp_pos = [s.pos0 + PAGE * i for r in reqs for s in r.spans for i in range(s.n_pages)]
    assert blk.tolist() == exp_blk
    assert ppos.tolist() == exp_pos
    qpos = B[B[L_OFF_QPOS]: B[L_OFF_QPOS] + L.total_query]
    assert qpos.tolist() == [r.query_pos0 + t for r in reqs for t in range(r.n_query)]
    # every (request, kv head, pair of 128-row tiles) appears once in the attention work list
    g = cfg.hq // cfg.hkv
    items = B[B[L_OFF_ATTN]: B[L_OFF_ATTN] + 4 * B[L_N_ATTN]].reshape(-1, 4)
    REQ = B[L_OFF_REQ]
    # per (request, tile pair): key-range splits and the first partial slot (pair records)
    pair_base = [int(B[REQ + 20 * b + 19]) for b in range(len(reqs))]
    n_pairs = [-(-r.n_rows * g // 256) for r in reqs]
    PR = B[L_OFF_PAIR]
    nsplit = {(b, t): int(B[PR + 2 * (pair_base[b] + t)]) for b in range(len(reqs)) for t in range(n_pairs[b])}
    want = {(b, h, t, s) for b in range(len(reqs)) for h in range(cfg.hkv)
            for t in range(n_pairs[b]) for s in range(nsplit[(b, t)])}
    got = {tuple(x) for x in items.tolist()}
    assert got == want and len(items) == len(want)
    assert all(1 <= n <= 16 for n in nsplit.values())
    assert B[L_N_PAIRS] == sum(n_pairs)
    # partial slots: consecutive blocks of Hkv * nsplit for the split pairs, in pair order
    slot = 0
    for b in range(len(reqs)):
        for t in range(n_pairs[b]):
            if nsplit[(b, t)] > 1:
                assert B[PR + 2 * (pair_base[b] + t) + 1] == slot
                slot += cfg.hkv * nsplit[(b, t)]
    assert B[34] == slot                     # partial slots in total
    # combine items: exactly the split (request, kv head, pair)s
    comb = B[B[L_OFF_COMB]: B[L_OFF_COMB] + 4 * B[L_N_COMB]].reshape(-1, 4)
    assert {tuple(x[:3]) for x in comb.tolist()} == {(b, h, t) for (b, t), n in nsplit.items() if n > 1
                                                      for h in range(cfg.hkv)}
    # importance runs {req, first tile, kv head | chunk pair << 16, tiles}: every (request, key
    # tile, kv head, pair of 256-row query chunks) once; a request with at most two chunks has one
    # pair, which keeps them both resident
    imp = B[B[L_OFF_IMP]: B[L_OFF_IMP] + 4 * B[L_N_IMP]].reshape(-1, 4)
    covered = [(int(q), t, int(hc) & 0xFFFF, int(hc) >> 16) for q, t0, hc, nt in imp.tolist()
               for t in range(t0, t0 + nt)]

    def pairs(r):
        chunks = -(-r.n_query * g // 256)
        return -(-chunks // 2) if chunks > 2 else 1
    assert sorted(covered) == sorted((b, t, h, p) for b, r in enumerate(reqs)
                                     for t in range(-(-r.n_cached // 128)) for h in range(cfg.hkv)
                                     for p in range(pairs(r)))
    assert all(nt >= 1 for nt in imp[:, 3])


def test_shared_pages_at_two_offsets_in_one_batch():
    # one physical span, two requests, logical offsets 0 and 2048 (position-free reuse)
    b = small_custom_batch([(0, 2, 0, 3)], n_query=4, extra_requests=[([(0, 2, 2048, 3)], 4, 2080)])
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, 4096, device="cpu")
    B = _blob(L)
    blk = B[B[L_OFF_BLOCK]: B[L_OFF_BLOCK] + 4].tolist()
    ppos = B[B[L_OFF_PAGEPOS]: B[L_OFF_PAGEPOS] + 4].tolist()
    assert blk == [0, 1, 0, 1]
    assert ppos == [0, 16, 2048, 2064]


def _try_build(spans_list, hq=4, hkv=2, d=64, n_phys=8, max_pos=4096, n_query=4, qpos=None):
    lib = _lib.load()
    reqs = (_lib.RequestDesc * len(spans_list))()
    keep = []
    for i, spans in enumerate(spans_list):
        arr = (_lib.SpanDesc * max(1, len(spans)))(*[_lib.SpanDesc(*s) for s in spans])
        keep.append(arr)
        end = max([s[2] + 16 * s[1] for s in spans] + [0])
        reqs[i] = _lib.RequestDesc(len(spans), arr, n_query, end if qpos is None else qpos)
    dims = _lib.Dims(hq, hkv, d, n_phys, max_pos)
    n = ctypes.c_int64(0)
    st = lib.pcf_layout_words(reqs, len(spans_list), ctypes.byref(dims), ctypes.byref(n))
    if st != 0:
        return st
    buf = (ctypes.c_int32 * n.value)()
    return lib.pcf_layout_build(reqs, len(spans_list), ctypes.byref(dims), buf, n.value)


def test_layout_validation():
    ok = [(0, 2, 0, 3), (2, 1, 40, 16)]
    assert _try_build([ok]) == 0
    assert _try_build([[(0, 2, 10, 3), (2, 1, 30, 0)]]) == -1       # overlapping positions
    assert _try_build([[(0, 2, 10, 3), (2, 1, 5, 0)]]) == -1        # positions not increasing
    assert _try_build([[(0, 2, 4090, 3)]]) == -1                     # beyond max_pos
    assert _try_build([[(7, 2, 0, 3)]]) == -1                        # outside the pool
    assert _try_build([[(0, 0, 0, 0)]]) == -1                        # empty span
    assert _try_build([[(0, 1, 0, 17)]]) == -1                       # k > span length
    assert _try_build([[(0, 1, 0, -1)]]) == -1                       # k < 0
    assert _try_build([ok], qpos=20) == -1                           # query inside the spans
    assert _try_build([ok], hq=6, hkv=4) == -2                       # Hq % Hkv != 0
    assert _try_build([ok], d=96) == -2                              # head_dim not 64/128
    assert _try_build([ok], hq=256, hkv=1) == -2                     # group larger than a tile
    assert _try_build([[]]) == 0                                     # a request with no spans
    lib = _lib.load()
    dims = _lib.Dims(4, 2, 64, 8, 4096)
    n = ctypes.c_int64(0)
    assert lib.pcf_layout_words(None, 1, ctypes.byref(dims), ctypes.byref(n)) == -1
    assert lib.pcf_layout_build(None, 1, ctypes.byref(dims), None, 0) == -1


def test_layout_too_small_buffer_and_query():
    lib = _lib.load()
    spans = (_lib.SpanDesc * 1)(_lib.SpanDesc(0, 2, 0, 3))
    reqs = (_lib.RequestDesc * 1)(_lib.RequestDesc(1, spans, 4, 32))
    dims = _lib.Dims(4, 2, 64, 8, 4096)
    n = ctypes.c_int64(0)
    assert lib.pcf_layout_words(reqs, 1, ctypes.byref(dims), ctypes.byref(n)) == 0
    small = (ctypes.c_int32 * (n.value - 1))()
    assert lib.pcf_layout_build(reqs, 1, ctypes.byref(dims), small, n.value - 1) == -1
    buf = (ctypes.c_int32 * n.value)()
    assert lib.pcf_layout_build(reqs, 1, ctypes.byref(dims), buf, n.value) == 0
    v = ctypes.c_int64(0)
    assert lib.pcf_layout_query(buf, 8, ctypes.byref(v)) == 0 and v.value == 32
    assert lib.pcf_layout_query(buf, 99, ctypes.byref(v)) == -1
    ws = ctypes.c_size_t(0)
    assert lib.pcf_score_workspace_bytes(buf, ctypes.byref(ws)) == 0 and ws.value > 0
    assert lib.pcf_attention_workspace_bytes(buf, ctypes.byref(ws)) == 0 and ws.value > 0


def test_work_lists_are_planned_for_the_named_sm_count():
    lib = _lib.load()
    spans = (_lib.SpanDesc * 2)(_lib.SpanDesc(0, 64, 0, 100), _lib.SpanDesc(64, 64, 1024, 100))
    reqs = (_lib.RequestDesc * 1)(_lib.RequestDesc(2, spans, 64, 2048))

    def build(n_sms):
        dims = _lib.Dims(32, 8, 128, 128, 4096, n_sms)
        n = ctypes.c_int64(0)
        st = lib.pcf_layout_words(reqs, 1, ctypes.byref(dims), ctypes.byref(n))
        if st != 0:
            return st, None
        buf = (ctypes.c_int32 * n.value)()
        assert lib.pcf_layout_build(reqs, 1, ctypes.byref(dims), buf, n.value) == 0
        return 0, np.frombuffer(buf, dtype=np.int32).copy()

    assert build(4097)[0] == -1
    _, default = build(0)
    _, gb300 = build(152)
    _, small = build(8)
    assert default[37] == 152 and small[37] == 8
    assert np.array_equal(default, gb300)
    # one request of 144 rows: on a small GPU its key range needs no split across CTAs
    assert small[L_N_ATTN] <= default[L_N_ATTN]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_device_calls_fail_loudly_without_gpu():
    b = small_custom_batch([(0, 2, 0, 3)], n_query=4)
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, 4096, device="cpu")
    imp = torch.empty(32, dtype=torch.float32)
    sel = torch.empty(3, dtype=torch.int32)
    ex = torch.empty(2, dtype=torch.int16)
    rp = torch.empty(7, dtype=torch.int32)
    with pytest.raises(pcf.PcfError) as e:
        lib = _lib.load()
        _lib.check("pcf_select_topk", lib.pcf_select_topk(
            ctypes.byref(L.ref), ctypes.c_void_p(imp.data_ptr()), ctypes.c_void_p(sel.data_ptr()),
            ctypes.c_void_p(ex.data_ptr()), ctypes.c_void_p(rp.data_ptr()), None))
    assert e.value.status == -7


def test_variant_entry_points_validate_before_touching_a_device(lib):
    """Global Top-N, key norms and anchor packing reject bad arguments on the host (no device
    needed): null buffers, and anchor counts that do not fill whole pages."""
    PCF_ERR_INVALID_ARG = -1
    b = small_custom_batch([(0, 2, 0, 3), (2, 2, 32, 5)], n_query=4)
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, 4096, device="cpu")
    ref = ctypes.byref(L.ref)
    assert lib.pcf_select_topn_global(ref, None, None, None, None, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_key_norms(ref, None, None, None) == PCF_ERR_INVALID_ARG
    # 3 + 5 anchors: not a whole page
    assert lib.pcf_pack_anchor_pages(ref, None, None, None, None, None, None) == PCF_ERR_INVALID_ARG
    b16 = small_custom_batch([(0, 2, 0, 16), (2, 2, 32, 0)], n_query=4)
    L16 = pcf.Layout(b16.requests, b16.hq, b16.hkv, b16.d, b16.n_phys_pages, 4096, device="cpu")
    # whole pages, but no buffers
    assert lib.pcf_pack_anchor_pages(ctypes.byref(L16.ref), None, None, None, None, None, None) == PCF_ERR_INVALID_ARG
    # prefetch: K pools required, V pools both or neither
    k = torch.zeros(b.n_phys_pages * b.hkv * 16 * b.d, dtype=torch.bfloat16)
    pk = ctypes.c_void_p(k.data_ptr())
    assert lib.pcf_prefetch_pool_pages(ref, None, None, pk, None, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_prefetch_pool_pages(ref, pk, pk, pk, None, None) == PCF_ERR_INVALID_ARG


def test_variant_layouts_build_with_the_expected_totals():
    """The layouts the variants use: the whole span pool as one query-less request (anchor key
    norms), anchor counts in whole pages (anchor packing), and the probe (one span of anchor pages
    per request, nothing recomputed, the query right after the anchors)."""
    from oracle import method
    from workload import Request, Span
    cfg = CONFIGS["concurrent_reuse"]
    pps = cfg.span_len // PAGE
    n_phys = cfg.pool_spans * pps
    pool = [Request(spans=[Span(i * pps, pps, i * cfg.span_len, 0) for i in range(cfg.pool_spans)], n_query=0,
                    query_pos0=cfg.pool_spans * cfg.span_len)]
    L = pcf.Layout(pool, cfg.hq, cfg.hkv, cfg.d, n_phys, cfg.pool_spans * cfg.span_len + 1, device="cpu")
    assert (L.total_tokens, L.total_sel, L.total_rows, L.total_query) == (cfg.pool_spans * cfg.span_len, 0, 0, 0)
    reqs = make_layout(cfg)
    anchors = [Request(spans=[Span(s.phys_first_page, s.n_pages, s.pos0, method.anchor_count(6, s.n_pages * PAGE))
                              for s in r.spans], n_query=r.n_query, query_pos0=r.query_pos0) for r in reqs]
    A = pcf.Layout(anchors, cfg.hq, cfg.hkv, cfg.d, n_phys, max(r.query_pos0 + r.n_query for r in reqs) + 1,
                   device="cpu")
    per_req = [r.n_sel for r in anchors]
    assert all(n % PAGE == 0 for n in per_req) and A.total_sel == sum(per_req)
    base = np.concatenate([[0], np.cumsum(per_req)])
    probe = [Request(spans=[Span(int(base[i]) // PAGE, r.n_sel // PAGE, 0, 0)], n_query=r.n_query, query_pos0=r.n_sel)
             for i, r in enumerate(anchors)]
    P = pcf.Layout(probe, cfg.hq, cfg.hkv, cfg.d, A.total_sel // PAGE,
                   max(r.n_sel + r.n_query for r in anchors) + 1, device="cpu")
    assert P.total_tokens == A.total_sel and P.total_sel == 0
    assert P.total_rows == sum(r.n_query for r in reqs)


def test_wait_limit_check_validates_on_the_host(lib):
    """The bounded-wait check rejects limits outside [1000, 2e8] cycles and a null or misaligned
    flag before looking for a device."""
    PCF_ERR_INVALID_ARG = -1
    flag = torch.zeros(2, dtype=torch.int32)
    p = flag.data_ptr()
    assert lib.pcf_wait_limit_check(999, ctypes.c_void_p(p), None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_wait_limit_check(200000001, ctypes.c_void_p(p), None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_wait_limit_check(100000, None, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_wait_limit_check(100000, ctypes.c_void_p(p + 2), None) == PCF_ERR_INVALID_ARG


def test_score_layers_validates_on_the_host(lib):
    """All-layer scoring rejects a layer count outside [1, 4096], missing pointer arrays and a
    null layer pool before looking for a device."""
    PCF_ERR_INVALID_ARG = -1
    b = small_custom_batch([(0, 2, 0, 3)], n_query=4)
    L = pcf.Layout(b.requests, b.hq, b.hkv, b.d, b.n_phys_pages, 4096, device="cpu")
    ref = ctypes.byref(L.ref)
    buf = torch.zeros(4096, dtype=torch.float32)
    p = ctypes.c_void_p(buf.data_ptr())
    arr = (ctypes.c_void_p * 2)(buf.data_ptr(), buf.data_ptr())
    nul = (ctypes.c_void_p * 2)(buf.data_ptr(), None)
    assert lib.pcf_score_layers(ref, 0, arr, arr, p, p, p, p, 1 << 20, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_score_layers(ref, 4097, arr, arr, p, p, p, p, 1 << 20, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_score_layers(ref, 2, None, arr, p, p, p, p, 1 << 20, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_score_layers(ref, 2, arr, nul, p, p, p, p, 1 << 20, None) == PCF_ERR_INVALID_ARG
    assert lib.pcf_score_layers(ref, 2, arr, arr, p, None, p, p, 1 << 20, None) == PCF_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["concurrent_reuse", "batch70b"])
def test_paged_attention_workspace_holds_no_copy_of_the_cached_keys(name):
    """The paged attention keeps no copy of the cached keys or values: its workspace is the
    compacted call's minus (at least) the rotated K and copied V of every kept cached token."""
    from workload import CONFIGS, make_layout
    cfg = CONFIGS[name]
    reqs = make_layout(cfg)
    L = pcf.Layout(reqs, cfg.hq, cfg.hkv, cfg.d, cfg.pool_spans * cfg.span_len // 16,
                   max(r.query_pos0 + r.n_query for r in reqs) + 1, device="cpu")
    paged, compact = L.attention_paged_workspace_bytes(), L.attention_workspace_bytes()
    kv_copy = 2 * cfg.hkv * cfg.d * 2 * (L.total_tokens - L.total_sel)
    assert compact - paged >= kv_copy
    # scoring: the rotated copy of every cached key (fp16, every kv head) is gone as well
    assert L.score_workspace_bytes() - L.score_paged_workspace_bytes() >= cfg.hkv * cfg.d * 2 * L.total_tokens


def test_paged_attention_workspace_does_not_grow_with_cached_tokens():
    """Same rows, four times the cached tokens: the compacted call's workspace grows with them; the
    paged call's, apart from the split partials (which follow the work plan's key-range splits),
    grows only by a 4-byte counter per page."""
    small = small_custom_batch([(0, 8, 0, 16)], n_query=32, hq=8, hkv=2, d=128, theta=5e5, n_phys_pages=64)
    big = small_custom_batch([(0, 32, 0, 16)], n_query=32, hq=8, hkv=2, d=128, theta=5e5, n_phys_pages=64)
    Ls = pcf.Layout(small.requests, 8, 2, 128, 64, 4096, device="cpu")
    Lb = pcf.Layout(big.requests, 8, 2, 128, 64, 4096, device="cpu")
    L_ATTN_SLOTS = 34

    def without_partials(L):   # 256 partial rows per slot: d bf16 values and a (max, sum) pair
        return L.attention_paged_workspace_bytes() - int(L.host[L_ATTN_SLOTS]) * 256 * (128 * 2 + 8)

    assert without_partials(Lb) <= without_partials(Ls) + 4 * (Lb.total_pages - Ls.total_pages) + 4096
    assert Lb.attention_workspace_bytes() > 3 * Ls.attention_workspace_bytes() // 2
