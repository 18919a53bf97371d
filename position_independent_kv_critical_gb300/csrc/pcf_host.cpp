// Host side of the C ABI: status strings, recompute counts, the RoPE table and the layout blob.
//
// The layout follows the position-free cache of MiniPIC (section 2.1): keys stay unrotated in
// shared physical pages and every request only supplies logical positions pi(j) through a block
// table, so the same physical page may appear in several requests at different offsets
// (section 1, "concurrency barrier").  Spans are page-aligned (section 2.2, "Padding").
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "../../include/pcf.h"
#include "layout_format.h"

using namespace pcf;

extern "C" const char* pcf_status_string(pcf_status s) {
    switch (s) {
        case PCF_OK: return "ok";
        case PCF_ERR_INVALID_ARG: return "invalid argument";
        case PCF_ERR_UNSUPPORTED: return "unsupported shape (head_dim must be 64 or 128; Hq/Hkv must divide 128)";
        case PCF_ERR_CUDA: return "CUDA call failed";
        case PCF_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
        case PCF_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PCF_ERR_DEVICE_BOUNDS: return "a kernel met an out-of-range index";
        case PCF_ERR_NO_DEVICE: return "no sm_103 device is current";
        default: return "unknown status";
    }
}

extern "C" int32_t pcf_k_from_percent(int32_t pct, int32_t span_len) {
    if (pct < 0 || span_len < 0) return -1;
    const int64_t num = (int64_t)pct * (int64_t)span_len;
    return (int32_t)((num + 99) / 100);
}

extern "C" pcf_status pcf_rope_table_init(float* table, int32_t head_dim, double theta,
                                          int32_t max_pos) {
    if (!table || !(theta > 0.0) || max_pos < kPage || max_pos > kMaxPosLimit)
        return PCF_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PCF_ERR_UNSUPPORTED;
    const int half = head_dim / 2;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) inv[i] = std::pow(theta, -2.0 * i / head_dim);
    for (int64_t p = 0; p < max_pos; ++p) {
        float* row = table + p * (int64_t)head_dim;
        for (int i = 0; i < half; ++i) {
            const double a = (double)p * inv[i];
            row[2 * i] = (float)std::cos(a);
            row[2 * i + 1] = (float)std::sin(a);
        }
    }
    return PCF_OK;
}

namespace {

struct Plan {
    int64_t words = 0;
    int32_t total_tokens = 0, total_query = 0, total_rows = 0, total_sel = 0, total_pages = 0;
    int32_t n_spans = 0, max_tokens = 0, max_rows = 0, max_query = 0, total_ktiles = 0;
    int32_t n_attn = 0, n_lse = 0, n_imp = 0, lse_slots = 0, max_span_len = 0;
    int32_t n_comb = 0, attn_slots = 0;
    std::vector<int32_t> lse_chunks, nsplit;
};

inline int32_t cdiv(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }

pcf_status validate(const pcf_request_desc* reqs, int32_t n_reqs, const pcf_dims* dims, Plan* plan) {
    if (!reqs || !dims || n_reqs < 1 || n_reqs > (1 << 20)) return PCF_ERR_INVALID_ARG;
    const pcf_dims& d = *dims;
    if (d.n_q_heads < 1 || d.n_kv_heads < 1 || d.n_phys_pages < 0 || d.max_pos < kPage ||
        d.max_pos > kMaxPosLimit)
        return PCF_ERR_INVALID_ARG;
    if (d.head_dim != 64 && d.head_dim != 128) return PCF_ERR_UNSUPPORTED;
    if (d.n_q_heads % d.n_kv_heads != 0) return PCF_ERR_UNSUPPORTED;
    const int g = d.n_q_heads / d.n_kv_heads;
    if (g > kTileRows || kTileRows % g != 0) return PCF_ERR_UNSUPPORTED;

    int64_t tot_tok = 0, tot_q = 0, tot_rows = 0, tot_sel = 0, tot_spans = 0, tot_kt = 0;
    int64_t base_lse_ctas = 0, base_attn_ctas = 0;
    for (int b = 0; b < n_reqs; ++b) {
        const pcf_request_desc& r = reqs[b];
        if (r.n_spans < 0 || r.n_query < 0 || (r.n_spans > 0 && !r.spans)) return PCF_ERR_INVALID_ARG;
        int64_t last_end = -1;   // first position after the previous span
        int64_t n_tok = 0, n_sel = 0;
        for (int s = 0; s < r.n_spans; ++s) {
            const pcf_span_desc& sp = r.spans[s];
            if (sp.n_pages < 1 || sp.phys_first_page < 0 ||
                (int64_t)sp.phys_first_page + sp.n_pages > d.n_phys_pages)
                return PCF_ERR_INVALID_ARG;
            if (sp.pos0 < 0 || (last_end >= 0 && sp.pos0 < last_end)) return PCF_ERR_INVALID_ARG;
            const int64_t len = (int64_t)sp.n_pages * kPage;
            if (sp.pos0 + len > d.max_pos) return PCF_ERR_INVALID_ARG;
            if (sp.k < 0 || sp.k > len) return PCF_ERR_INVALID_ARG;
            last_end = sp.pos0 + len;
            n_tok += len;
            n_sel += sp.k;
            plan->max_span_len = std::max<int32_t>(plan->max_span_len, (int32_t)len);
        }
        if (r.query_pos0 < 0 || (last_end >= 0 && r.query_pos0 < last_end)) return PCF_ERR_INVALID_ARG;
        if ((int64_t)r.query_pos0 + r.n_query > d.max_pos) return PCF_ERR_INVALID_ARG;
        tot_tok += n_tok;
        tot_q += r.n_query;
        tot_rows += n_sel + r.n_query;
        tot_sel += n_sel;
        tot_spans += r.n_spans;
        const int32_t nkt = cdiv(n_tok / kPage, kPagesPerTile);
        tot_kt += nkt;
        if (nkt > 0 && r.n_query > 0)
            base_lse_ctas += (int64_t)d.n_kv_heads * cdiv((int64_t)r.n_query * g, kTileRows * kQTilesPerCta);
        base_attn_ctas += (int64_t)d.n_kv_heads * cdiv((n_sel + r.n_query) * g, kTileRows * kQTilesPerCta);
        plan->max_tokens = std::max<int32_t>(plan->max_tokens, (int32_t)n_tok);
        plan->max_rows = std::max<int32_t>(plan->max_rows, (int32_t)(n_sel + r.n_query));
        plan->max_query = std::max<int32_t>(plan->max_query, r.n_query);
    }
    // every row of every [rows][H][d] tensor must stay addressable with 32-bit row indices
    const int64_t lim = (int64_t)1 << 30;
    if (tot_tok >= lim || tot_rows * g >= lim || tot_q * g >= lim) return PCF_ERR_INVALID_ARG;
    if ((int64_t)d.n_phys_pages * d.n_kv_heads * kPage >= ((int64_t)1 << 31)) return PCF_ERR_INVALID_ARG;

    plan->total_tokens = (int32_t)tot_tok;
    plan->total_query = (int32_t)tot_q;
    plan->total_rows = (int32_t)tot_rows;
    plan->total_sel = (int32_t)tot_sel;
    plan->total_pages = (int32_t)(tot_tok / kPage);
    plan->n_spans = (int32_t)tot_spans;
    plan->total_ktiles = (int32_t)tot_kt;

    // key-chunk split of the LSE pass: aim for ~kLseTargetCtas CTAs in total
    const int32_t want = base_lse_ctas > 0 ? cdiv(kLseTargetCtas, base_lse_ctas) : 1;
    // key-range split of the attention: only batches too small to fill the GPU with tile pairs
    const int32_t want_split = base_attn_ctas > 0 ? std::min<int64_t>(kMaxSplits, cdiv(kAttnTargetCtas, base_attn_ctas)) : 1;
    plan->lse_chunks.assign(n_reqs, 0);
    plan->nsplit.assign(n_reqs, 1);
    int64_t n_attn = 0, n_lse = 0, n_imp = 0, slots = 0, n_comb = 0, attn_slots = 0;
    for (int b = 0; b < n_reqs; ++b) {
        const pcf_request_desc& r = reqs[b];
        int64_t n_tok = 0, n_sel = 0;
        for (int s = 0; s < r.n_spans; ++s) {
            n_tok += (int64_t)r.spans[s].n_pages * kPage;
            n_sel += r.spans[s].k;
        }
        const int32_t nkt = cdiv(n_tok / kPage, kPagesPerTile);
        const int64_t rows = n_sel + r.n_query;
        const int64_t npairs = cdiv(rows * g, kTileRows * kQTilesPerCta);
        const int32_t max_tiles = nkt + cdiv(rows, kTileKeys);   // key tiles the last pair sees
        const int32_t ns = std::max(1, std::min<int32_t>(want_split, max_tiles / kMinTilesPerSplit));
        plan->nsplit[b] = ns;
        n_attn += (int64_t)d.n_kv_heads * npairs * ns;
        if (ns > 1) {
            n_comb += (int64_t)d.n_kv_heads * npairs;
            attn_slots += (int64_t)d.n_kv_heads * npairs * ns;
        }
        if (nkt > 0 && r.n_query > 0) {
            const int32_t tpc = cdiv(nkt, std::max(1, std::min(want, nkt)));
            const int32_t chunks = cdiv(nkt, tpc);
            plan->lse_chunks[b] = chunks;
            n_lse += (int64_t)d.n_kv_heads * cdiv((int64_t)r.n_query * g, kTileRows * kQTilesPerCta) * chunks;
            slots += (int64_t)r.n_query * d.n_q_heads * chunks;
        }
        if (nkt > 0) n_imp += (int64_t)nkt * d.n_kv_heads;
    }
    if (n_attn >= lim || n_lse >= lim || n_imp >= lim || slots >= lim || attn_slots >= lim / 256)
        return PCF_ERR_INVALID_ARG;
    plan->n_comb = (int32_t)n_comb;
    plan->attn_slots = (int32_t)attn_slots;
    plan->n_attn = (int32_t)n_attn;
    plan->n_lse = (int32_t)n_lse;
    plan->n_imp = (int32_t)n_imp;
    plan->lse_slots = (int32_t)slots;

    plan->words = L_HEADER + (int64_t)n_reqs * R_STRIDE + tot_spans * S_STRIDE +
                  2 * (int64_t)plan->total_pages + kItemWords * (n_attn + n_lse + n_imp + n_comb) + tot_q;
    if (plan->words >= ((int64_t)1 << 31)) return PCF_ERR_INVALID_ARG;
    return PCF_OK;
}

}  // namespace

extern "C" pcf_status pcf_layout_words(const pcf_request_desc* reqs, int32_t n_reqs,
                                       const pcf_dims* dims, int64_t* n_words) {
    if (!n_words) return PCF_ERR_INVALID_ARG;
    Plan plan;
    pcf_status st = validate(reqs, n_reqs, dims, &plan);
    if (st != PCF_OK) return st;
    *n_words = plan.words;
    return PCF_OK;
}

extern "C" pcf_status pcf_layout_build(const pcf_request_desc* reqs, int32_t n_reqs,
                                       const pcf_dims* dims, int32_t* blob, int64_t n_words) {
    if (!blob) return PCF_ERR_INVALID_ARG;
    Plan plan;
    pcf_status st = validate(reqs, n_reqs, dims, &plan);
    if (st != PCF_OK) return st;
    if (n_words < plan.words) return PCF_ERR_INVALID_ARG;
    std::memset(blob, 0, sizeof(int32_t) * (size_t)plan.words);
    const pcf_dims& d = *dims;
    const int g = d.n_q_heads / d.n_kv_heads;

    int32_t* H = blob;
    H[L_MAGIC] = kMagic;
    H[L_WORDS] = (int32_t)plan.words;
    H[L_N_REQS] = n_reqs;
    H[L_HQ] = d.n_q_heads;
    H[L_HKV] = d.n_kv_heads;
    H[L_D] = d.head_dim;
    H[L_N_PHYS] = d.n_phys_pages;
    H[L_MAX_POS] = d.max_pos;
    H[L_TOTAL_TOKENS] = plan.total_tokens;
    H[L_TOTAL_QUERY] = plan.total_query;
    H[L_TOTAL_ROWS] = plan.total_rows;
    H[L_TOTAL_SEL] = plan.total_sel;
    H[L_TOTAL_PAGES] = plan.total_pages;
    H[L_N_SPANS] = plan.n_spans;
    H[L_MAX_TOKENS] = plan.max_tokens;
    H[L_MAX_ROWS] = plan.max_rows;
    H[L_MAX_QUERY] = plan.max_query;
    H[L_TOTAL_KTILES] = plan.total_ktiles;
    H[L_N_ATTN_ITEMS] = plan.n_attn;
    H[L_N_LSE_ITEMS] = plan.n_lse;
    H[L_N_IMP_ITEMS] = plan.n_imp;
    H[L_LSE_SLOTS] = plan.lse_slots;
    H[L_GROUP] = g;
    H[L_MAX_SPAN_LEN] = plan.max_span_len;
    H[L_N_COMB] = plan.n_comb;
    H[L_ATTN_SLOTS] = plan.attn_slots;

    int64_t off = L_HEADER;
    H[L_OFF_REQ] = (int32_t)off;    off += (int64_t)n_reqs * R_STRIDE;
    H[L_OFF_SPAN] = (int32_t)off;   off += (int64_t)plan.n_spans * S_STRIDE;
    H[L_OFF_BLOCK] = (int32_t)off;  off += plan.total_pages;
    H[L_OFF_PAGEPOS] = (int32_t)off; off += plan.total_pages;
    H[L_OFF_ATTN] = (int32_t)off;   off += (int64_t)kItemWords * plan.n_attn;
    H[L_OFF_LSE] = (int32_t)off;    off += (int64_t)kItemWords * plan.n_lse;
    H[L_OFF_IMP] = (int32_t)off;    off += (int64_t)kItemWords * plan.n_imp;
    H[L_OFF_QPOS] = (int32_t)off;   off += plan.total_query;
    H[L_OFF_COMB] = (int32_t)off;   off += (int64_t)kItemWords * plan.n_comb;

    int32_t* REQ = blob + H[L_OFF_REQ];
    int32_t* SPN = blob + H[L_OFF_SPAN];
    int32_t* BLK = blob + H[L_OFF_BLOCK];
    int32_t* PPOS = blob + H[L_OFF_PAGEPOS];
    int32_t* QPOS = blob + H[L_OFF_QPOS];

    struct AttnItem { int32_t req, kvh, qt, split; int64_t cost; int64_t order; };
    std::vector<AttnItem> attn;
    attn.reserve(plan.n_attn);
    int32_t* LSE = blob + H[L_OFF_LSE];
    int32_t* IMP = blob + H[L_OFF_IMP];
    int32_t* COMB = blob + H[L_OFF_COMB];
    int64_t n_lse = 0, n_imp = 0, n_comb = 0;
    int32_t slot_base = 0;

    int32_t tok_base = 0, q_base = 0, row_base = 0, sel_base = 0, span_base = 0, kt_base = 0;
    int32_t lse_base = 0;
    for (int b = 0; b < n_reqs; ++b) {
        const pcf_request_desc& r = reqs[b];
        int32_t* R = REQ + (int64_t)b * R_STRIDE;
        int32_t n_pages = 0, n_sel = 0;
        for (int s = 0; s < r.n_spans; ++s) {
            const pcf_span_desc& sp = r.spans[s];
            int32_t* S = SPN + (int64_t)(span_base + s) * S_STRIDE;
            S[S_REQ] = b;
            S[S_PAGE_OFF] = n_pages;
            S[S_N_PAGES] = sp.n_pages;
            S[S_K] = sp.k;
            S[S_SEL_OFF] = n_sel;
            S[S_POS0] = sp.pos0;
            S[S_PHYS_FIRST] = sp.phys_first_page;
            for (int p = 0; p < sp.n_pages; ++p) {
                BLK[tok_base / kPage + n_pages + p] = sp.phys_first_page + p;
                PPOS[tok_base / kPage + n_pages + p] = sp.pos0 + p * kPage;
            }
            n_pages += sp.n_pages;
            n_sel += sp.k;
        }
        const int32_t n_tok = n_pages * kPage;
        const int32_t n_rows = n_sel + r.n_query;
        const int32_t nkt = cdiv(n_pages, kPagesPerTile);
        R[R_N_PAGES] = n_pages;
        R[R_TOK_BASE] = tok_base;
        R[R_PAGE_BASE] = tok_base / kPage;
        R[R_Q_BASE] = q_base;
        R[R_ROW_BASE] = row_base;
        R[R_SEL_BASE] = sel_base;
        R[R_QUERY_POS0] = r.query_pos0;
        R[R_N_SPANS] = r.n_spans;
        R[R_SPAN_BASE] = span_base;
        R[R_N_QUERY] = r.n_query;
        R[R_N_SEL] = n_sel;
        R[R_N_ROWS] = n_rows;
        R[R_LSE_BASE] = lse_base;
        R[R_LSE_CHUNKS] = plan.lse_chunks[b];
        R[R_KTILE_BASE] = kt_base;
        R[R_N_KTILES] = nkt;
        const int32_t ns = plan.nsplit[b];
        R[R_NSPLIT] = ns;
        R[R_SLOT_BASE] = slot_base;
        for (int t = 0; t < r.n_query; ++t) QPOS[q_base + t] = r.query_pos0 + t;

        // attention work: one item per (kv head, pair of 128-row tiles); rows pack the g heads of a
        // token
        const int32_t toks_per_item = kQTilesPerCta * (kTileRows / g);
        const int32_t n_qt = cdiv((int64_t)n_rows * g, kTileRows * kQTilesPerCta);
        R[R_NPAIRS] = n_qt;
        if (ns > 1) slot_base += d.n_kv_heads * n_qt * ns;
        for (int32_t qt = 0; qt < n_qt; ++qt) {
            const int64_t last_row = std::min<int64_t>((int64_t)(qt + 1) * toks_per_item, n_rows) - 1;
            // estimated visible keys: query rows see everything, recomputed rows about the
            // fraction of the context before them
            int64_t cost;
            if (last_row >= n_sel) cost = (int64_t)n_tok + n_rows;
            else cost = ((int64_t)(last_row + 1) * (n_tok + n_sel)) / std::max<int64_t>(1, n_sel);
            for (int32_t h = 0; h < d.n_kv_heads; ++h) {
                for (int32_t sp = 0; sp < ns; ++sp)
                    attn.push_back({b, h, qt, sp, cost / ns, (int64_t)attn.size()});
                if (ns > 1) {
                    int32_t* it = COMB + kItemWords * n_comb++;
                    it[0] = b; it[1] = h; it[2] = qt; it[3] = 0;
                }
            }
        }
        // LSE work: (kv head, query tile pair, key chunk)
        if (plan.lse_chunks[b] > 0) {
            const int32_t n_lqt = cdiv((int64_t)r.n_query * g, kTileRows * kQTilesPerCta);
            for (int32_t h = 0; h < d.n_kv_heads; ++h)
                for (int32_t qt = 0; qt < n_lqt; ++qt)
                    for (int32_t c = 0; c < plan.lse_chunks[b]; ++c) {
                        int32_t* it = LSE + kItemWords * n_lse++;
                        it[0] = b; it[1] = h; it[2] = qt; it[3] = c;
                    }
            lse_base += r.n_query * d.n_q_heads * plan.lse_chunks[b];
        }
        // importance work: (key tile, kv head)
        for (int32_t t = 0; t < nkt; ++t)
            for (int32_t h = 0; h < d.n_kv_heads; ++h) {
                int32_t* it = IMP + kItemWords * n_imp++;
                it[0] = b; it[1] = t; it[2] = h; it[3] = 0;
            }
        tok_base += n_tok;
        q_base += r.n_query;
        row_base += n_rows;
        sel_base += n_sel;
        span_base += r.n_spans;
        kt_base += nkt;
    }
    std::stable_sort(attn.begin(), attn.end(), [](const AttnItem& a, const AttnItem& b) {
        return a.cost > b.cost;
    });
    int32_t* ATT = blob + H[L_OFF_ATTN];
    for (size_t i = 0; i < attn.size(); ++i) {
        ATT[kItemWords * i + 0] = attn[i].req;
        ATT[kItemWords * i + 1] = attn[i].kvh;
        ATT[kItemWords * i + 2] = attn[i].qt;
        ATT[kItemWords * i + 3] = attn[i].split;
    }
    return PCF_OK;
}

extern "C" pcf_status pcf_layout_query(const int32_t* blob, int32_t field, int64_t* value) {
    if (!blob || !value || blob[L_MAGIC] != kMagic || field < 1 || field >= L_HEADER)
        return PCF_ERR_INVALID_ARG;
    *value = blob[field];
    return PCF_OK;
}
