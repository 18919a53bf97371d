"""fp64 CPU oracle of the cache-fusion hot path (test infrastructure only).

Steps, in the order the pages give them:

1. the request's cached keys/values are read from the pool pages in logical order; key j sits at
   logical position pi(j) (MiniPIC, section 2.1: "logical position of cached key j in the current
   request"; one physical block serves requests at different offsets, section 1 "concurrency
   barrier");
2. critical-layer profiling: attention of the query tokens over the cached keys only, each key
   rotated explicitly at pi(j), each query at its own position, softmax over all cached keys of
   the request, weights summed over heads and query tokens (QCFuse, section 2B; second summary
   Phase 3);
3. Top-N selection of the tokens to recompute, per span, ties to the lower index (QCFuse 2B),
   or over the whole request with the same budget (the pages' own global Top-N);
4. fused attention of the recomputed rows and the query rows over the merged key set: cached keys
   minus the recomputed tokens, plus the fresh rows at their positions, causal on logical
   position (QCFuse 2C and Phase 4; second summary section 3 "strictly keeps causal constraints";
   MiniPIC 2.1 score equation).

Offline, before any request (QCFuse 2A, second summary Phase 1): each span's anchor tokens, the
few with the highest key norm; at request time (Phase 2) the query attends over the request's
anchors put in front of it as a prefix.

Readings where the pages are silent: rotate-half RoPE pairing; softmax
over the request's cached keys only for scoring; a plain sum over heads and query tokens; query
head h reads kv head floor(h / g); a key is visible to a row iff its logical position is <= the
row's; scale 1/sqrt(d); no temperature, cap or sink.

All inputs are converted to fp64 exactly (bf16 -> fp64 is exact).  Nothing here is blocked, fused
or reordered beyond the definitions; matmul, exp and sort are library steps.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

from .rope import rotate

PAGE = 16


def k_from_percent(pct: int, length: int) -> int:
    """Tokens recomputed in a span of ``length`` at ``pct`` percent: ceil(pct*length/100) in
    integers (the pages fix no rounding; reading used throughout)."""
    return -((-int(pct) * int(length)) // 100)


def request_cached(spans, k_pool: np.ndarray, v_pool: np.ndarray
                   ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Cached keys / values of one request in logical order and their logical positions.

    ``spans``: sequence of objects with ``phys_first_page``, ``n_pages`` and ``pos0``.
    ``k_pool`` / ``v_pool``: [P_phys][Hkv][16][d].  Returns K~ [N][Hkv][d], V [N][Hkv][d] (fp64)
    and pi [N] (int64)."""
    hkv, d = k_pool.shape[1], k_pool.shape[3]
    pages = [s.phys_first_page + i for s in spans for i in range(s.n_pages)]
    if not pages:
        z = np.zeros((0, hkv, d))
        return z, z.copy(), np.zeros((0,), dtype=np.int64)
    kp = np.asarray(k_pool, dtype=np.float64)[pages]          # [np][Hkv][16][d]
    vp = np.asarray(v_pool, dtype=np.float64)[pages]
    K = kp.transpose(0, 2, 1, 3).reshape(-1, hkv, d)
    V = vp.transpose(0, 2, 1, 3).reshape(-1, hkv, d)
    pos = np.concatenate([s.pos0 + np.arange(s.n_pages * PAGE, dtype=np.int64) for s in spans])
    return K, V, pos


def _softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax with max subtraction; rows that are entirely -inf give zeros."""
    m = np.max(s, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m)
    tot = e.sum(axis=-1, keepdims=True)
    return np.divide(e, tot, out=np.zeros_like(e), where=tot > 0)


def score_request(q: np.ndarray, q_pos: np.ndarray, K: np.ndarray, k_pos: np.ndarray,
                  theta: float) -> np.ndarray:
    """Importance of each cached token for one request.

    imp[j] = sum_h sum_t softmax_j( (R_{pos(t)} q_{t,h}) . (R_{pi(j)} k~_{j,h/g}) / sqrt(d) )

    q [T][Hq][d], q_pos [T], K [N][Hkv][d] unrotated, k_pos [N].  Returns imp [N] fp64."""
    T, hq, d = q.shape
    N, hkv = K.shape[0], K.shape[1]
    g = hq // hkv
    imp = np.zeros(N, dtype=np.float64)
    if N == 0 or T == 0:
        return imp
    qr = rotate(q, q_pos, theta)      # explicit rotation of each query at its position
    kr = rotate(K, k_pos, theta)      # explicit rotation of each cached key at pi(j)
    scale = 1.0 / math.sqrt(d)
    for h in range(hq):
        s = (qr[:, h, :] @ kr[:, h // g, :].T) * scale          # [T][N]
        imp += _softmax_rows(s).sum(axis=0)
    return imp


def score_layers_request(q_layers: Sequence[np.ndarray], q_pos: np.ndarray, K_layers: Sequence[np.ndarray],
                         k_pos: np.ndarray, theta: float) -> Tuple[np.ndarray, np.ndarray]:
    """Importance taken at every layer instead of one critical layer (the all-layer comparison
    point of QCFuse, section 4 "Resultados", QCAll; the last layer alone is QCLast): layer l's
    query tokens attend over layer l's cached keys exactly as in ``score_request``, and the
    request's importance is the plain sum of the layers' importances (the pages name no rule for
    combining layers; a mean would rank the tokens the same way).

    q_layers[l] [T][Hq][d], K_layers[l] [N][Hkv][d] unrotated; positions are the request's, the
    same at every layer.  Returns (per-layer importance [L][N], their sum over layers [N])."""
    per = np.stack([score_request(q, q_pos, K, k_pos, theta) for q, K in zip(q_layers, K_layers)]) \
        if len(q_layers) else np.zeros((0, len(k_pos)))
    return per, per.sum(axis=0)


def select_topk_request(imp: np.ndarray, span_lens: Sequence[int], span_k: Sequence[int]
                        ) -> np.ndarray:
    """Per span: the k_s request-local token indices with the largest importance, ties to the
    lower index, returned in ascending index order, spans concatenated.

    ``imp`` is taken exactly as given (pass fp32 values to take the decision in fp32)."""
    imp = np.asarray(imp, dtype=np.float64)
    out: List[np.ndarray] = []
    off = 0
    for L, k in zip(span_lens, span_k):
        vals = imp[off: off + L]
        order = np.lexsort((np.arange(L), -vals))    # primary key: -value, then index
        out.append(np.sort(order[:k]).astype(np.int64) + off)
        off += L
    return np.concatenate(out) if out else np.zeros((0,), dtype=np.int64)


def select_topn_global_request(imp: np.ndarray, n_sel: int) -> np.ndarray:
    """QCFuse, section 2B (Top-N tokens of the whole context) and its Phase 3 summary: the n_sel
    request-local token indices with the largest importance over all of the request's cached
    tokens, ties to the lower index, in ascending index order.  The budget n_sel is the sum of the
    spans' k, so only the placement across spans differs from the per-span selection.

    ``imp`` is taken exactly as given (pass fp32 values to take the decision in fp32)."""
    imp = np.asarray(imp, dtype=np.float64)
    order = np.lexsort((np.arange(imp.shape[0]), -imp))    # primary key: -value, then index
    return np.sort(order[:n_sel]).astype(np.int64)


def key_norms(K: np.ndarray) -> np.ndarray:
    """QCFuse, section 2A (anchor extraction) and Phase 1: the magnitude of each cached token's
    key, read here as the Euclidean norm of its unrotated key over all kv heads and dimensions,
    ``K`` [N][Hkv][d] -> [N] (fp64).  Rotation preserves the norm, so the cached (position-free)
    key gives the same value as the key at any position."""
    K = np.asarray(K, dtype=np.float64)
    return np.sqrt((K * K).reshape(K.shape[0], -1).sum(axis=1))


def select_anchors_request(norms: np.ndarray, span_lens: Sequence[int], span_m: Sequence[int]
                           ) -> np.ndarray:
    """QCFuse, section 2A: per span, the m_s tokens with the highest key norm are its anchors
    (a small share of the span's tokens), ties to the lower index, ascending; the same per-span
    selection as the recompute Top-N, on the key norms instead of the importance."""
    return select_topk_request(norms, span_lens, span_m)


def anchor_count(pct: int, length: int) -> int:
    """Anchors of a span of ``length`` tokens at ``pct`` percent, rounded up to whole pages of 16:
    16 * ceil(pct * length / 1600).  The pages give only "a small share"; whole pages let the
    anchors be packed into pages of their own and read like any cached span."""
    return PAGE * (-((-int(pct) * int(length)) // (100 * PAGE)))


def anchor_probe_request(q: np.ndarray, k: np.ndarray, v: np.ndarray, K_anchor: np.ndarray,
                         V_anchor: np.ndarray, theta: float) -> np.ndarray:
    """QCFuse, section 2A (injection) and Phase 2: the anchors are put in front of the query as a
    prefix, at positions 0 .. A-1 in span order, the query tokens follow at A .. A+T-1, and each
    query token attends over the anchors and, causally, over the query tokens; fp64 [T][Hq][d].
    ``q`` [T][Hq][d], ``k``/``v`` [T][Hkv][d] the query tokens' own projections, ``K_anchor``/
    ``V_anchor`` [A][Hkv][d] the anchors' cached (unrotated) keys and values."""
    A, T = K_anchor.shape[0], q.shape[0]
    return fused_attention_request(q, k, v, A + np.arange(T, dtype=np.int64), K_anchor, V_anchor,
                                   np.arange(A, dtype=np.int64), np.zeros((0,), dtype=np.int64), theta)


def row_positions(sel: np.ndarray, k_pos: np.ndarray, n_query: int, query_pos0: int) -> np.ndarray:
    """Logical positions of a request's rows: the selected tokens (ascending), then the query."""
    return np.concatenate([k_pos[sel], query_pos0 + np.arange(n_query, dtype=np.int64)])


def exclusion_masks(sel: np.ndarray, n_pages: int) -> np.ndarray:
    """uint16 per logical page: bit r set iff token 16*page + r is recomputed."""
    m = np.zeros(n_pages, dtype=np.uint32)
    for j in np.asarray(sel, dtype=np.int64):
        m[j // PAGE] |= np.uint32(1) << np.uint32(j % PAGE)
    return m.astype(np.uint16)


def gather_rows(src_rows: np.ndarray, sel: np.ndarray) -> np.ndarray:
    """Rows of the selected tokens, in selection order (the recompute batch input)."""
    return np.asarray(src_rows)[np.asarray(sel, dtype=np.int64)]


def fused_attention_request(q_fresh: np.ndarray, k_fresh: np.ndarray, v_fresh: np.ndarray,
                            row_pos: np.ndarray, K: np.ndarray, V: np.ndarray, k_pos: np.ndarray,
                            sel: np.ndarray, theta: float,
                            rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Attention output for a request's rows (or the subset ``rows``), fp64 [rows][Hq][d].

    Keys = cached tokens not in ``sel`` (at pi(j)) followed by every fresh row (at row_pos); key u
    is visible to row r iff pos(u) <= row_pos[r]."""
    n_rows, hq, d = q_fresh.shape
    hkv = k_fresh.shape[1]
    g = hq // hkv
    if rows is None:
        rows = np.arange(n_rows)
    rows = np.asarray(rows, dtype=np.int64)
    keep = np.ones(K.shape[0], dtype=bool)
    keep[np.asarray(sel, dtype=np.int64)] = False
    key_pos = np.concatenate([k_pos[keep], row_pos]).astype(np.int64)
    k_all = np.concatenate([rotate(K[keep], k_pos[keep], theta), rotate(k_fresh, row_pos, theta)])
    v_all = np.concatenate([np.asarray(V, dtype=np.float64)[keep],
                            np.asarray(v_fresh, dtype=np.float64)])
    qr = rotate(q_fresh[rows], row_pos[rows], theta)
    visible = key_pos[None, :] <= row_pos[rows][:, None]          # [R][Nk]
    scale = 1.0 / math.sqrt(d)
    out = np.zeros((rows.shape[0], hq, d), dtype=np.float64)
    for h in range(hq):
        s = (qr[:, h, :] @ k_all[:, h // g, :].T) * scale
        s = np.where(visible, s, -np.inf)
        out[:, h, :] = _softmax_rows(s) @ v_all[:, h // g, :]
    return out


def full_prefill(q: np.ndarray, k: np.ndarray, v: np.ndarray, pos: np.ndarray,
                 theta: float) -> np.ndarray:
    """Plain causal prefill of n tokens at positions ``pos``: every token attends to every token
    at a position <= its own.  Written row by row, separately from the fused path, as the
    reference that 100 % recompute must reproduce.  q [n][Hq][d], k/v [n][Hkv][d]."""
    n, hq, d = q.shape
    g = hq // k.shape[1]
    qr = rotate(q, pos, theta)
    kr = rotate(k, pos, theta)
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros((n, hq, d), dtype=np.float64)
    for r in range(n):
        vis = np.nonzero(pos <= pos[r])[0]
        for h in range(hq):
            logits = kr[vis, h // g, :] @ qr[r, h, :] / math.sqrt(d)
            w = np.exp(logits - logits.max())
            out[r, h, :] = (w / w.sum()) @ v[vis, h // g, :]
    return out


# ----------------------------------------------------------------------------------------------
# Whole-batch drivers (duck-typed request objects: .spans [.phys_first_page .n_pages .pos0 .k],
# .n_query, .query_pos0)
# ----------------------------------------------------------------------------------------------

def batch_score(requests, q_query: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                theta: float, req_ids: Optional[Sequence[int]] = None) -> List[np.ndarray]:
    """Importance per request (fp64).  ``q_query`` [sum T][Hq][d] concatenated over requests."""
    qb = np.cumsum([0] + [r.n_query for r in requests])
    out = []
    ids = range(len(requests)) if req_ids is None else req_ids
    for b in ids:
        r = requests[b]
        K, _, kpos = request_cached(r.spans, k_pool, v_pool)
        q = np.asarray(q_query[qb[b]: qb[b + 1]], dtype=np.float64)
        qpos = r.query_pos0 + np.arange(r.n_query, dtype=np.int64)
        out.append(score_request(q, qpos, K, kpos, theta))
    return out


def batch_select(requests, imps: Sequence[np.ndarray], req_ids: Optional[Sequence[int]] = None
                 ) -> List[np.ndarray]:
    ids = range(len(requests)) if req_ids is None else req_ids
    return [select_topk_request(imp, [s.n_pages * PAGE for s in requests[b].spans],
                                [s.k for s in requests[b].spans])
            for imp, b in zip(imps, ids)]
