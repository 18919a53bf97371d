// Host side of the C ABI: status strings, recompute counts, the RoPE table and the layout blob.
//
// The layout follows the position-free cache of MiniPIC (section 2.1): keys stay unrotated in
// shared physical pages and every request only supplies logical positions pi(j) through a block
// table, so the same physical page may appear in several requests at different offsets
// (section 1, "concurrency barrier").  Spans are page-aligned (section 2.2, "Padding").
#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <queue>
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
        case PCF_ERR_DEVICE_RANGE: return "a rotated query or key is outside the fp16 range (|x| > 65504)";
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
    int32_t n_comb = 0, attn_slots = 0, n_pairs = 0, imp_tiles = 1;
    int32_t n_sms = kDefaultSms;        // SMs the work lists are planned for
    std::vector<int32_t> lse_chunks;
    std::vector<int32_t> pair_base;     // per request: first pair record
    std::vector<int32_t> pair_tiles;    // per pair record: estimated key tiles of the pair
    std::vector<int32_t> pair_split;    // per pair record: key-range splits
};

inline int32_t cdiv(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }

// Estimated finishing time (in key tiles) of CTAs with the given costs on n_sms SMs that take
// one CTA each at a time, launched in decreasing cost order (the order of the work lists).
double lpt_makespan(std::vector<double>& costs, int32_t n_sms) {
    std::sort(costs.begin(), costs.end(), std::greater<double>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> sm;
    for (int i = 0; i < n_sms; ++i) sm.push(0.0);
    double end = 0.0;
    for (double c : costs) {
        const double t = sm.top() + c;
        sm.pop();
        sm.push(t);
        end = std::max(end, t);
    }
    return end;
}

// Key-range splits per work unit (a unit runs once per kv head: `copies` CTAs) that minimise the
// estimated finishing time when a CTA costs `overhead` tiles plus its share of the unit's tiles
// and any split adds `combine` tiles (the merge of the partial results).  Batches with enough
// units to fill the GPU several times are not split.
void choose_splits(const std::vector<int32_t>& tiles, int32_t copies, double overhead, double combine,
                   int32_t max_split, int32_t n_sms, std::vector<int32_t>* splits) {
    splits->assign(tiles.size(), 1);
    if (tiles.empty() || (int64_t)tiles.size() * copies >= 4 * n_sms) return;
    int32_t max_t = 1;
    for (int32_t t : tiles) max_t = std::max(max_t, t);
    double best = 0.0;
    int32_t best_c = max_t;
    std::vector<double> costs;
    for (int32_t c = max_t; c >= 1; --c) {   // candidate tiles per split, largest first
        costs.clear();
        bool any = false;
        for (int32_t t : tiles) {
            const int32_t sp = std::max(1, std::min({cdiv(t, c), max_split, t}));
            any = any || sp > 1;
            costs.insert(costs.end(), (size_t)copies * sp, overhead + (double)t / sp);
        }
        const double end = lpt_makespan(costs, n_sms) + (any ? combine : 0.0);
        if (c == max_t || end < best - 1e-9) {
            best = end;
            best_c = c;
        }
    }
    for (size_t i = 0; i < tiles.size(); ++i)
        (*splits)[i] = std::max(1, std::min({cdiv(tiles[i], best_c), max_split, tiles[i]}));
}

// Prologue + epilogue of an attention CTA in key tiles, and of the merge of split results.
constexpr double kAttnCtaOverhead = 1.5;
constexpr double kAttnCombineCost = 2.0;
constexpr double kLseCtaOverhead = 2.0;
constexpr double kImpCtaOverhead = 1.0;

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
    if (d.n_sms > 4096) return PCF_ERR_INVALID_ARG;
    plan->n_sms = d.n_sms > 0 ? d.n_sms : kDefaultSms;

    int64_t tot_tok = 0, tot_q = 0, tot_rows = 0, tot_sel = 0, tot_spans = 0, tot_kt = 0;
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

    // Attention work units: (request, pair of 128-row query tiles), each run once per kv head.  A
    // pair sees the request's cached tiles (eight pages each; a recomputed token's fresh key takes
    // its cached copy's place) up to its last row's position and the tiles of query rows up to its
    // last row.  Rows are selected tokens in position order, then query tokens; before the
    // selection is known, a selected row is only known to lie inside its span, so the span's end
    // bounds its cached tiles.
    plan->pair_base.assign(n_reqs, 0);
    plan->pair_tiles.clear();
    for (int b = 0; b < n_reqs; ++b) {
        const pcf_request_desc& r = reqs[b];
        int64_t n_sel = 0, n_pg = 0;
        std::vector<int64_t> cum_k(1, 0), cum_pages(1, 0);
        for (int s = 0; s < r.n_spans; ++s) {
            n_sel += r.spans[s].k;
            n_pg += r.spans[s].n_pages;
            cum_k.push_back(n_sel);
            cum_pages.push_back(n_pg);
        }
        const int32_t nkt = cdiv(n_pg, kPagesPerTile);
        const int64_t rows = n_sel + r.n_query;
        const int64_t npairs = cdiv(rows * g, kTileRows * kQTilesPerCta);
        const int64_t toks_per_pair = (int64_t)kQTilesPerCta * (kTileRows / g);
        plan->pair_base[b] = (int32_t)plan->pair_tiles.size();
        size_t s = 0;
        for (int64_t p = 0; p < npairs; ++p) {
            const int64_t last = std::min<int64_t>((p + 1) * toks_per_pair, rows) - 1;
            int32_t nct = nkt, nft = 0;
            if (last < n_sel) {
                while (s + 1 < cum_k.size() && cum_k[s + 1] <= last) ++s;
                nct = cdiv(cum_pages[s + 1], kPagesPerTile);
            } else {
                nft = (int32_t)((last - n_sel) / kTileKeys) + 1;
            }
            plan->pair_tiles.push_back(nct + nft);
        }
    }
    choose_splits(plan->pair_tiles, d.n_kv_heads, kAttnCtaOverhead, kAttnCombineCost, kMaxSplits, plan->n_sms,
                  &plan->pair_split);
    // LSE pass: units (request, query tile pair) over all cached tiles, split into key chunks
    std::vector<int32_t> lse_split;
    {
        std::vector<int32_t> tiles, copies;
        for (int b = 0; b < n_reqs; ++b) {
            const pcf_request_desc& r = reqs[b];
            int64_t n_pg = 0;
            for (int s = 0; s < r.n_spans; ++s) n_pg += r.spans[s].n_pages;
            const int32_t nkt = cdiv(n_pg, kPagesPerTile);
            if (nkt > 0 && r.n_query > 0)
                for (int32_t p = 0; p < cdiv((int64_t)r.n_query * g, kTileRows * kQTilesPerCta); ++p) tiles.push_back(nkt);
        }
        std::vector<int32_t> sp;
        choose_splits(tiles, d.n_kv_heads, kLseCtaOverhead, 0.0, kMaxSplits, plan->n_sms, &sp);
        size_t u = 0;
        for (int b = 0; b < n_reqs; ++b) {
            const pcf_request_desc& r = reqs[b];
            int64_t n_pg = 0;
            for (int s = 0; s < r.n_spans; ++s) n_pg += r.spans[s].n_pages;
            const int32_t nkt = cdiv(n_pg, kPagesPerTile);
            int32_t want = 1;
            if (nkt > 0 && r.n_query > 0) {
                want = sp[u];   // every pair of a request has the same tiles, hence the same split
                u += cdiv((int64_t)r.n_query * g, kTileRows * kQTilesPerCta);
            }
            lse_split.push_back(want);
        }
    }
    plan->lse_chunks.assign(n_reqs, 0);
    int64_t n_attn = 0, n_lse = 0, n_imp = 0, slots = 0, n_comb = 0, attn_slots = 0;
    // importance pass: CTAs over runs of key tiles of one kv head; run lengths by the same
    // estimate as the attention splits (a CTA costs about one step more than its tiles)
    {
        std::vector<int32_t> tiles, sp;
        for (int b = 0; b < n_reqs; ++b) {
            int64_t n_pg = 0;
            for (int s = 0; s < reqs[b].n_spans; ++s) n_pg += reqs[b].spans[s].n_pages;
            if (n_pg > 0) tiles.push_back(cdiv(n_pg, kPagesPerTile));
        }
        choose_splits(tiles, d.n_kv_heads, kImpCtaOverhead, 0.0, 1 << 20, plan->n_sms, &sp);
        int32_t run = 1;
        for (size_t u = 0; u < tiles.size(); ++u) run = std::max(run, cdiv(tiles[u], sp[u]));
        plan->imp_tiles = run;
    }
    for (int b = 0; b < n_reqs; ++b) {
        const pcf_request_desc& r = reqs[b];
        int64_t n_tok = 0;
        for (int s = 0; s < r.n_spans; ++s) n_tok += (int64_t)r.spans[s].n_pages * kPage;
        const int32_t nkt = cdiv(n_tok / kPage, kPagesPerTile);
        const int32_t p0 = plan->pair_base[b];
        const int32_t p1 = b + 1 < n_reqs ? plan->pair_base[b + 1] : (int32_t)plan->pair_tiles.size();
        for (int32_t p = p0; p < p1; ++p) {
            const int32_t ns = plan->pair_split[p];
            n_attn += (int64_t)d.n_kv_heads * ns;
            if (ns > 1) {
                n_comb += d.n_kv_heads;
                attn_slots += (int64_t)d.n_kv_heads * ns;
            }
        }
        if (nkt > 0 && r.n_query > 0) {
            const int32_t tpc = cdiv(nkt, std::max(1, std::min(lse_split[b], nkt)));
            const int32_t chunks = cdiv(nkt, tpc);
            plan->lse_chunks[b] = chunks;
            n_lse += (int64_t)d.n_kv_heads * cdiv((int64_t)r.n_query * g, kTileRows * kQTilesPerCta) * chunks;
            slots += (int64_t)r.n_query * d.n_q_heads * chunks;
        }
        if (nkt > 0) n_imp += (int64_t)cdiv(nkt, plan->imp_tiles) * d.n_kv_heads * imp_chunk_pairs(r.n_query, g);
    }
    plan->n_pairs = (int32_t)plan->pair_tiles.size();
    if (n_attn >= lim || n_lse >= lim || n_imp >= lim || slots >= lim || attn_slots >= lim / 256)
        return PCF_ERR_INVALID_ARG;
    plan->n_comb = (int32_t)n_comb;
    plan->attn_slots = (int32_t)attn_slots;
    plan->n_attn = (int32_t)n_attn;
    plan->n_lse = (int32_t)n_lse;
    plan->n_imp = (int32_t)n_imp;
    plan->lse_slots = (int32_t)slots;

    plan->words = L_HEADER + (int64_t)n_reqs * R_STRIDE + tot_spans * S_STRIDE +
                  2 * (int64_t)plan->total_pages + kItemWords * (n_attn + n_lse + n_imp + n_comb) + tot_q +
                  (int64_t)P_STRIDE * plan->n_pairs;
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
    H[L_TOTAL_VALID] = plan.total_tokens - plan.total_sel;
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
    H[L_N_PAIRS] = plan.n_pairs;
    H[L_N_SMS] = plan.n_sms;

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
    H[L_OFF_PAIR] = (int32_t)off;   off += (int64_t)P_STRIDE * plan.n_pairs;

    int32_t* REQ = blob + H[L_OFF_REQ];
    int32_t* SPN = blob + H[L_OFF_SPAN];
    int32_t* BLK = blob + H[L_OFF_BLOCK];
    int32_t* PPOS = blob + H[L_OFF_PAGEPOS];
    int32_t* QPOS = blob + H[L_OFF_QPOS];

    struct AttnItem { int32_t req, kvh, qt, split; double cost; };
    std::vector<AttnItem> attn;
    attn.reserve(plan.n_attn);
    int32_t* LSE = blob + H[L_OFF_LSE];
    int32_t* IMP = blob + H[L_OFF_IMP];
    int32_t* PAIR = blob + H[L_OFF_PAIR];
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
        R[R_PAIR_BASE] = plan.pair_base[b];
        R[R_CBASE] = tok_base - sel_base;   // taking-part cached keys of the requests before
        for (int t = 0; t < r.n_query; ++t) QPOS[q_base + t] = r.query_pos0 + t;

        // attention work: per (pair of 128-row tiles, kv head), one item per key-range split; rows
        // pack the g heads of a token
        const int32_t n_qt = cdiv((int64_t)n_rows * g, kTileRows * kQTilesPerCta);
        R[R_NPAIRS] = n_qt;
        for (int32_t qt = 0; qt < n_qt; ++qt) {
            const int32_t pr = plan.pair_base[b] + qt;
            const int32_t ns = plan.pair_split[pr];
            PAIR[P_STRIDE * pr + P_NSPLIT] = ns;
            PAIR[P_STRIDE * pr + P_SLOT_BASE] = slot_base;
            if (ns > 1) slot_base += d.n_kv_heads * ns;
            const double cost = kAttnCtaOverhead + (double)plan.pair_tiles[pr] / ns;
            for (int32_t h = 0; h < d.n_kv_heads; ++h) {
                for (int32_t sp = 0; sp < ns; ++sp) attn.push_back({b, h, qt, sp, cost});
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
        // importance work: (run of key tiles, kv head, pair of query chunks); the request's tiles
        // are cut into ceil(nkt / imp_tiles) runs of near-equal length, and a run's chunk pairs are
        // neighbours in the list so that their CTAs run together and share the key tiles in L2
        if (nkt > 0) {
            const int32_t runs = cdiv(nkt, plan.imp_tiles);
            const int32_t n_cp = imp_chunk_pairs(r.n_query, g);
            for (int32_t u = 0; u < runs; ++u) {
                const int32_t t0 = (int32_t)((int64_t)u * nkt / runs), t1 = (int32_t)((int64_t)(u + 1) * nkt / runs);
                for (int32_t h = 0; h < d.n_kv_heads; ++h)
                    for (int32_t cp = 0; cp < n_cp; ++cp) {
                        int32_t* it = IMP + kItemWords * n_imp++;
                        it[0] = b; it[1] = t0; it[2] = h | (cp << 16); it[3] = t1 - t0;
                    }
            }
        }
        tok_base += n_tok;
        q_base += r.n_query;
        row_base += n_rows;
        sel_base += n_sel;
        span_base += r.n_spans;
        kt_base += nkt;
    }
    // Hand-out order.  With a few items per SM (small batches): longest first, so that the CTAs
    // finishing last hold short items.  With many: grouped by (request, kv head) unit -- units in
    // decreasing total cost, each unit's items longest first -- so that the CTAs running at one
    // time share a few units' K/V tiles in L2 (a unit's items all read prefixes of the same keys)
    // instead of each streaming its own unit's from DRAM; the dynamic hand-out still balances the
    // end, where the last unit's short items run.
    if ((int64_t)attn.size() >= 8LL * plan.n_sms) {
        std::vector<double> ucost((size_t)n_reqs * d.n_kv_heads, 0.0);
        for (const AttnItem& a : attn) ucost[(size_t)a.req * d.n_kv_heads + a.kvh] += a.cost;
        std::stable_sort(attn.begin(), attn.end(), [&](const AttnItem& a, const AttnItem& b) {
            const double ua = ucost[(size_t)a.req * d.n_kv_heads + a.kvh];
            const double ub = ucost[(size_t)b.req * d.n_kv_heads + b.kvh];
            if (ua != ub) return ua > ub;
            if (a.req != b.req) return a.req < b.req;
            if (a.kvh != b.kvh) return a.kvh < b.kvh;
            return a.cost > b.cost;
        });
    } else {
        std::stable_sort(attn.begin(), attn.end(), [](const AttnItem& a, const AttnItem& b) {
            return a.cost > b.cost;
        });
    }
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
