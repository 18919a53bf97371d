// Word map of the layout blob built by pcf_layout_build and read by the kernels.
//
// The blob carries everything the position-free cache needs per batch (MiniPIC, section 2.1:
// per-request logical positions over shared physical blocks; section 2.2: spans padded to page
// boundaries): the block table (logical page -> physical page), the logical position of each
// page's first token, span and request records, and precomputed work lists so that no launch
// needs host-side knowledge beyond the header.
#pragma once
#include <stdint.h>

namespace pcf {

constexpr int32_t kMagic = 0x4C464350;   // "PCFL"
constexpr int kPage = 16;                // tokens per page
constexpr int kTileRows = 128;           // TMEM lanes = rows of one MMA tile
constexpr int kTileKeys = 128;           // keys per KV tile
constexpr int kQTilesPerCta = 2;         // 128-row query tiles sharing each rotated K/V tile
constexpr int kPagesPerTile = kTileKeys / kPage;
constexpr int kMaxPosLimit = 1 << 20;
constexpr int kItemWords = 4;
constexpr int kDefaultSms = 152;        // GB300's SM count: the plan's target when the caller names none
constexpr int kMaxSplits = 16;          // key-range splits of one attention (or LSE) work unit
constexpr int kImpQRows = 256;          // query rows of one importance chunk (the MMA's N)

// importance CTAs of a request per (run of key tiles, kv head): one per pair of query chunks (a
// CTA keeps its two chunks resident and streams its key tiles once)
#ifdef __CUDACC__
#define PCF_HOST_DEVICE __host__ __device__
#else
#define PCF_HOST_DEVICE
#endif
PCF_HOST_DEVICE inline int32_t imp_chunk_pairs(int64_t n_query, int32_t group) {
    const int64_t chunks = (n_query * group + kImpQRows - 1) / kImpQRows;
    return chunks > 2 ? (int32_t)((chunks + 1) / 2) : 1;
}

enum : int {
    L_MAGIC = 0, L_WORDS = 1, L_N_REQS = 2, L_HQ = 3, L_HKV = 4, L_D = 5, L_N_PHYS = 6,
    L_MAX_POS = 7, L_TOTAL_TOKENS = 8, L_TOTAL_QUERY = 9, L_TOTAL_ROWS = 10, L_TOTAL_SEL = 11,
    L_TOTAL_PAGES = 12, L_N_SPANS = 13, L_MAX_TOKENS = 14, L_MAX_ROWS = 15, L_MAX_QUERY = 16,
    L_TOTAL_KTILES = 17, L_N_ATTN_ITEMS = 18, L_N_LSE_ITEMS = 19, L_N_IMP_ITEMS = 20,
    L_LSE_SLOTS = 21, L_GROUP = 22, L_MAX_SPAN_LEN = 23,
    L_OFF_REQ = 24, L_OFF_SPAN = 25, L_OFF_BLOCK = 26, L_OFF_PAGEPOS = 27, L_OFF_ATTN = 28,
    L_OFF_LSE = 29, L_OFF_IMP = 30, L_OFF_QPOS = 31, L_OFF_COMB = 32, L_N_COMB = 33,
    L_ATTN_SLOTS = 34, L_OFF_PAIR = 35, L_N_PAIRS = 36,
    L_N_SMS = 37,         // SMs the work lists were planned for (the persistent grids use the device's own count)
    L_TOTAL_VALID = 38,   // cached keys that take part in the attention (not recomputed), all requests
    L_HEADER = 40
};

// per-request record
enum : int {
    R_N_PAGES = 0, R_TOK_BASE = 1, R_PAGE_BASE = 2, R_Q_BASE = 3, R_ROW_BASE = 4, R_SEL_BASE = 5,
    R_QUERY_POS0 = 6, R_N_SPANS = 7, R_SPAN_BASE = 8, R_N_QUERY = 9, R_N_SEL = 10, R_N_ROWS = 11,
    R_LSE_BASE = 12, R_LSE_CHUNKS = 13, R_KTILE_BASE = 14, R_N_KTILES = 15,
    R_CBASE = 17,       // first row of the request's taking-part cached keys in the compacted copy
    R_NPAIRS = 18,      // tile pairs of the request (per kv head)
    R_PAIR_BASE = 19,   // first pair record of the request
    R_STRIDE = 20
};

// per-span record
enum : int {
    S_REQ = 0, S_PAGE_OFF = 1, S_N_PAGES = 2, S_K = 3, S_SEL_OFF = 4, S_POS0 = 5,
    S_PHYS_FIRST = 6, S_STRIDE = 8
};

// per-(request, tile pair) record: the pair's attention key range is split over P_NSPLIT CTAs per
// kv head; with P_NSPLIT > 1 split s of kv head h writes partial slot P_SLOT_BASE + h*P_NSPLIT + s
enum : int { P_NSPLIT = 0, P_SLOT_BASE = 1, P_STRIDE = 2 };

// work items (kItemWords each)
//   attention : {req, kv head, q tile pair, key-range split}   largest estimated cost first, or
//               with many items per SM grouped by (req, kv head) unit
//   lse       : {req, kv head, q tile pair, key chunk}
//               (each chunk writes its rows' partial (max, sum); the importance kernel combines
//               a row's chunks into its log2-sum-exp)
// (a "q tile pair" p covers the 128-row query tiles 2p and 2p+1 of the request)
//   importance: {req, first key tile, kv head | chunk pair << 16, key tiles}
//   combine   : {req, kv head, q tile pair, 0}   pairs whose key range was split

}  // namespace pcf
