// Flash-style attention over the position-free paged cache (sm_103a).
//
// MiniPIC, section 2.1: cached keys k~_j stay unrotated in shared pages and are rotated at use time
// to the key's per-request logical position pi(j), so score(t, j) = (R_t q_t)^T (R_pi(j) k~_j) /
// sqrt(d).  Two ways to feed the cached keys:
//   compacted (PAGED = false): the rotation runs once per call (rope_rows_kernel in page gather
//     mode, into the call's workspace), which also leaves the recomputed tokens out and copies the
//     kept V rows beside the kept keys; a cached key tile is visited by every 256-row query block
//     of the request, and rotating it here costs more than writing and re-reading it once.
//   paged (PAGED = true): K and V tiles are TMA-copied from the pool pages through the block
//     table (one 16-row box per page), two rotator warps rotate each K tile in shared memory to
//     the request's positions before the MMA reads it, and the recomputed tokens' fresh K and V
//     rows overwrite their stale cached copies in place; no per-request copy of the cache.
// QCFuse, section 2C / Phase 4 (and the sparse attention kernel of its section 3): the recomputed
// tokens and the query tokens attend over the cached keys minus the recomputed ones plus the
// fresh rows, keeping causal order on logical positions.
//
// Persistent: one CTA per SM works through the item list (the first item is the CTA's own, the
// rest are handed out in list order, i.e. largest estimated cost first, through a global counter),
// so barriers, TMEM and tensor maps are set up once and the next item's Q tiles and first key
// tiles load while the current item drains.  Every barrier phase is counted across items.
//
// One item = two tiles A and B of 128 query rows each (a tile packs the g query heads of 128/g
// consecutive rows of one request, all sharing kv head `kvh`) against a range of the request's KV
// tiles of 128 keys; both tiles share every K and V tile:
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: S row from TMEM, causal cut,
//               online softmax (lazy rescale), P -> TMEM (over the S columns), O epilogue
//   warps 8/11  Q K^T issue for tile A / B (warp 8 also owns the TMEM allocation)
//   warps 12/13 P V issue for tile A / B.  Each key tile is processed in two 64-key halves and S
//               is double-buffered per query tile: P(q) V runs, then Q K(q+2) goes into the
//               buffer P(q) came from, while the softmax already works on S(q+1).  Four issuer
//               warps keep four independent MMA streams in flight; each runs its loop with the
//               whole warp converged and lane 0 issuing (measured faster than lane 0 alone)
//   warp  9     scheduler (takes the next item, counts its visible key tiles, publishes it in one
//               of two shared-memory slots), Q loads, K producer: rotated K tiles (compacted
//               cached or fresh, fp16, TMA) and, per key, its logical position; 2-stage ring
//   warp  10    V producer (TMA): compacted cached V tiles / fresh V tiles; 2-stage ring (paged:
//               the pool pages, then each recomputed token's fresh V row over its cached one)
//   warps 14/15 (paged only) rotators: each cached K tile rotated in place, the fresh keys of its
//               recomputed tokens written over their cached copies
// TMEM: tile t's two S half-buffers at columns t*128 + {0, 64} (64 fp32 columns = 64 keys each),
// O_A at [256,256+d), O_B at [384,384+d).  S = Q K^T is fp16 x fp16 (M=128, N=64 keys, K=d); P
// (bf16 pairs, 32 columns) overwrites the S half it came from and is the A operand of
// O += P V (M=128, N=d in one instruction, K=64 keys, V as an MN-major bf16 operand whose two
// 64-wide halves are 16 KB apart).
// Compacted, every cached key streamed takes part; paged, a recomputed token's slot holds its
// fresh row, and only the query rows form fresh tiles.  Key positions increase along the cached
// keys and along the fresh rows, and missing keys (past a ragged end) carry position kNoPos, so a
// row's visible keys in a tile are a prefix of it; only rows whose causal limit falls inside a
// tile need per-element masking.
// LSE mode (critical-layer scoring, pass 1) runs the same pipeline without P/V and writes the
// per-row running max and sum of one key chunk (the importance kernel combines a row's chunks).  Having no O, it gives each query tile two S
// buffers of a whole key tile (128 columns) and issues Q K^T with N = 128: half the MMA
// instructions of two 64-key halves.  Without pages the CTA has 12 warps, and each softmax thread
// loads its row's 128 scores at once and frees the S buffer before the arithmetic (with 14 warps'
// register budget it took them in two parts and held the buffer through the first part's);
// in paged scoring the two P V issuer warps, idle without P V, are the rotators and the scores
// come in two parts.
#pragma once
#include "layout_format.h"
#include "ptx.cuh"

namespace pcf {

// 14 warps (at most 4 per SM sub-partition, so each may hold 128 registers); the paged variant
// adds two rotator warps (16 warps, 128 registers each); scoring without pages needs no P V
// issuers and runs 12 warps (3 per sub-partition, up to 168 registers: room for a whole key
// tile's scores in the softmax)
constexpr int kAttnThreads = 448;
constexpr int kAttnThreadsPaged = 512;
// (the paged scoring pass needs no extra warps: its rotators are the two P V issuer warps, idle
// without P V)
template <bool PAGED, bool LSE = false> __host__ __device__ constexpr int attn_threads() {
    return PAGED && !LSE ? kAttnThreadsPaged : (LSE && !PAGED ? 384 : kAttnThreads);
}
constexpr int kWarpSoftB = 4;
constexpr int kWarpMma = 8;
constexpr int kWarpTma = 9;
constexpr int kWarpTmaV = 10;
constexpr int kWarpMmaB = 11;
constexpr int kWarpPvA = 12;
constexpr int kWarpPvB = 13;
constexpr int kWarpRot = 14;        // warps 14 and 15: rotation of the cached key tiles (scoring: 12, 13)
constexpr int kRotThreads = 64;
constexpr int kNoPos = 0x7FFFFFFF;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kTmemO = 256;     // O_A at 256, O_B at 384
constexpr int kStageRows = 32;       // fresh keys of a tile's recomputed tokens staged with the tile

struct AttnParams {
    const int32_t* layout;
    const int32_t* kpos_c;     // attention (compacted): logical position of every compacted cached key
    const int32_t* row_pos;    // attention: logical position of every row
    __nv_bfloat16* out;        // attention: [rows][Hq][D]
    float2* lse_part;          // LSE: (running max in log2 units, running sum); per request
                               //      [kv head][key chunk][query row x g]
    __nv_bfloat16* part_o;     // attention with a split key range: normalized partial O per slot
    float2* part_ml;           //   and its (running max, running sum) per row
    int32_t* sched;            // items handed out beyond the first gridDim.x; zero on entry
    // paged attention only:
    const uint16_t* excl;      // recompute bits per logical page
    const int32_t* cidx;       // per logical page, the request's kept tokens before it (plus the
                               //   request's base R_CBASE)
    const __half* k_rot;       // rotated fresh keys [Hkv][rows][D] fp16
    const __nv_bfloat16* v_fresh;   // fresh values [rows][Hkv][D]
    const float2* rope;        // (cos, sin) table [max_pos][D/2]
};

// One item as the scheduler hands it to the other roles.
struct AttnItem {
    int32_t req;               // < 0: no more items
    int32_t kvh, qpair, chunk; // chunk: LSE key chunk or attention key-range split
    int32_t n_ct, n_ft;        // visible cached / fresh key tiles of the pair (LSE: the chunk's tiles)
    int32_t t0;                // LSE: first key tile of the chunk
    int32_t jb, n_loc;         // this item's tiles: jb .. jb+n_loc-1 of the visible range
    // request / pair fields the other roles need, copied here so that they need no layout loads
    int32_t n_rows;            // the request's rows (LSE: its query tokens)
    int32_t row_base;          // first row of the request
    int32_t cbase;             // first compacted cached key of the request
    int32_t nsplit, slot_base; // attention: key-range splits of the pair and its first partial slot
    int32_t lse_base, lse_chunks;   // LSE: the request's partials and its chunks
    int32_t page_base;         // first logical page of the request (block table, positions, bits)
    int32_t n_pages, n_sel;    // the request's cached pages and recomputed tokens
    int32_t pad;
};

template <int D, bool LSE, bool PAGED = false>
struct AttnSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kQ = kTileRows * D * 2;          // one Q tile
    static constexpr int kK = kTileKeys * D * 2;
    static constexpr int kV = LSE ? 0 : kTileKeys * D * 2;
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kQTilesPerCta * kQ;
    static constexpr int oV = oK + kKStages * kK;
    // attention: per K stage, the fresh rotated keys of the tile's recomputed tokens (a block of
    // consecutive fresh rows, kStageRows of them, copied with the tile) and per page of the tile
    // its recompute bits and the rank of its first recomputed token
    static constexpr int kKst = PAGED && !LSE ? kStageRows * D * 2 : 0;
    static constexpr int oKst = oV + kVStages * kV;
    static constexpr int oKpos = oKst + kKStages * kKst;
    static constexpr int oMeta = oKpos + kKStages * kTileKeys * 4;   // (paged: 64 bytes a stage)
    // attention: per K stage, the (cos, sin) table rows the rotators start from: for each page of
    // the tile and each run of 2*D/16 of its keys, the row at the run's first position
    static constexpr int kRope = PAGED ? kPagesPerTile * 32 * 16 : 0;   // 32 float4 per page: 4 KB
    static constexpr int oRope = oMeta + kKStages * kPagesPerTile * 8;
    // attention: each softmax thread's output pointers, kept here across the tile loop
    static constexpr int oPark = oRope + kKStages * kRope;
    static constexpr int oBar = oPark + (PAGED && !LSE ? 256 * 16 : 0);
    static constexpr int kNumBars = 42;
    static constexpr int oMisc = oBar + kNumBars * 8;
    static constexpr int oItem = oMisc + 64;
    static constexpr int kBytes = oItem + 2 * (int)sizeof(AttnItem);
    static constexpr int kAlloc = kBytes + 1024;   // slack for 1024-byte alignment
    static_assert(kAlloc <= 232448, "more dynamic shared memory than a GB300 block can have");
    static constexpr uint32_t kTmemCols = 512;   // LSE: 2 tiles x 2 S buffers of 128 columns
};

// barrier slots
enum : int {
    B_Q_FULL = 0,      // the item's Q tiles landed (one phase per item)
    B_K_FULL = 1,      // [2] the stage holds the rotated fp16 K tile (every rotator thread arrives)
    B_K_EMPTY = 3,     // [2] both Q K^T that read the stage are done (one commit per issuer)
    B_KPOS_FREE = 5,   // [2] both softmax groups are done with the stage's key positions (256 arrivals)
    B_V_FULL = 7,      // [2] the stage holds the V tile, recomputed tokens' rows replaced (V warp)
    B_V_EMPTY = 9,     // [2] both P V that read the stage are done (one commit per issuer)
    B_S_FULL = 11,     // [4] per (Q tile, S half-buffer): S = Q K^T of a 64-key half landed (LSE:
                       //     of a whole key tile, per 128-column buffer)
    B_P_FULL = 15,     // [4] per (Q tile, S half-buffer): P written and O rescaled; in LSE mode:
                       //     the softmax has loaded that S buffer into registers
    B_PV_DONE = 19,    // [4] per (Q tile, S half-buffer): P V of that buffer's latest half is done
    B_O_DONE = 23,     // [2] per Q tile: the item's last P V is done (one phase per item)
    B_DRAIN = 25,      // [4] per issuer: its last MMA is done
    B_Q_EMPTY = 29,    // both Q K^T issuers are done with the item's Q tiles (one commit each)
    B_O_FREE = 30,     // [2] per Q tile: the softmax group has read the item's O (128 arrivals)
    B_ITEM_FULL = 32,  // [2] item slot written by the scheduler
    B_ITEM_EMPTY = 34, // [2] every consumer role has read the slot
    B_KPOS_FULL = 36,  // [2] the K tile's key positions written (every producer lane)
    B_KRAW_FULL = 38,  // [2] the K tile's copy landed (TMA; the rotators then make it B_K_FULL)
    B_VRAW_FULL = 40   // [2] the V tile's copy landed (TMA; the V producer then makes it B_V_FULL)
};

// In-place rotation of part of a cached K tile in a stage (128-byte swizzled rows, the two 64-wide
// halves 16 KB apart for d = 128): 16-byte chunk pair c -- dimensions 8c .. 8c+7 and d/2 + 8c .. --
// of the N keys key0 .. key0+N-1, which sit at consecutive positions.  (C, S, -S) hold the cos and
// sin of the thread's eight frequencies at key0's position as packed fp32 pairs (frequencies 8c+2e
// and 8c+2e+1 in pair e) and advance by one position step (STC, STS, -STS: the table's row 1) from
// key to key.  bf16 in, fp16 out; a value out of fp16 range raises the range error.
template <int D, int N>
__device__ __forceinline__ void rotate_page_keys(uint8_t* stage, int key0, int c, uint64_t (&C)[4], uint64_t (&S)[4],
                                                 uint64_t (&NS)[4], const uint64_t (&STC)[4],
                                                 const uint64_t (&STS)[4], const uint64_t (&NSTS)[4]) {
    const uint32_t o_hi = D == 128 ? 16384u : 0u;
    const int c_hi = D == 128 ? c : c + 4;
    float big = 0.f;
#pragma unroll 2
    for (int r = 0; r < N; ++r) {
        const int key = key0 + r;
        uint4* plo = reinterpret_cast<uint4*>(stage + sw128_off(key, c));
        uint4* phi = reinterpret_cast<uint4*>(stage + o_hi + sw128_off(key, c_hi));
        const uint4 a = *plo, b = *phi;
        const uint32_t ia[4] = {a.x, a.y, a.z, a.w}, ib[4] = {b.x, b.y, b.z, b.w};
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint64_t A = bf16x2_to_f2(ia[e]), B = bf16x2_to_f2(ib[e]);
            float y0, y1, z0, z1;
            f2_unpack(f2_fma(B, NS[e], f2_mul(A, C[e])), y0, y1);   // a cos - b sin
            f2_unpack(f2_fma(A, S[e], f2_mul(B, C[e])), z0, z1);    // b cos + a sin
            oa[e] = pack_f16x2_track(y0, y1, big);
            ob[e] = pack_f16x2_track(z0, z1, big);
        }
        *plo = make_uint4(oa[0], oa[1], oa[2], oa[3]);
        *phi = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        // the next key's angles: one position further
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint64_t cn = f2_fma(S[e], NSTS[e], f2_mul(C[e], STC[e]));
            const uint64_t sn = f2_fma(C[e], STS[e], f2_mul(S[e], STC[e]));
            NS[e] = f2_fma(C[e], NSTS[e], f2_mul(NS[e], STC[e]));
            C[e] = cn;
            S[e] = sn;
        }
    }
    if (big > kF16Limit) set_dev_error(kDevErrRange);
}

template <int D, bool LSE, bool PAGED>
__global__ void __launch_bounds__(attn_threads<PAGED, LSE>())
attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kcache,
            const __grid_constant__ CUtensorMap tm_vcache, const __grid_constant__ CUtensorMap tm_kfresh,
            const __grid_constant__ CUtensorMap tm_vfresh, const __grid_constant__ CUtensorMap tm_kstage,
            const AttnParams prm) {
    using SM = AttnSmem<D, LSE, PAGED>;
    constexpr int H = SM::kHalves;
    // slot readers: lane 0 of the 8 softmax warps and of the 2 Q K^T issuers (+ 2 P V issuers and
    // the V producer outside LSE mode)
    // (paged: and lane 0 of the two rotator warps)
    constexpr int kItemReaders = (LSE ? 10 : 13) + (PAGED ? 2 : 0);
    constexpr int kRot0 = LSE ? kWarpPvA : kWarpRot;   // first rotator warp (paged)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sQ = [&](int t) { return smem + SM::oQ + t * SM::kQ; };
    auto sKs = [&](int st) { return smem + SM::oK + st * SM::kK; };
    auto sVs = [&](int st) { return smem + SM::oV + st * SM::kV; };
    auto sKpos = [&](int st) { return reinterpret_cast<int32_t*>(smem + SM::oKpos) + st * kTileKeys; };
    auto sKst = [&](int st) { return smem + SM::oKst + st * SM::kKst; };
    auto sMeta = [&](int st) { return reinterpret_cast<int2*>(smem + SM::oMeta) + st * kPagesPerTile; };
    auto sRope = [&](int st) { return reinterpret_cast<float4*>(smem + SM::oRope + st * SM::kRope); };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::oBar);
    int32_t* misc = reinterpret_cast<int32_t*>(smem + SM::oMisc);
    // misc: [0] tmem base, [4] abort
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    AttnItem* slots = reinterpret_cast<AttnItem*>(smem + SM::oItem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* L = prm.layout;
    const int32_t* items = L + (LSE ? L[L_OFF_LSE] : L[L_OFF_ATTN]);
    const int n_items = LSE ? L[L_N_LSE_ITEMS] : L[L_N_ATTN_ITEMS];
    const int Hq = L[L_HQ], g = L[L_GROUP];
    const int toks_per_tile = kTileRows / g;

    if (tid == 0) {
        mbar_init(&bars[B_Q_FULL], 1);
        mbar_init(&bars[B_Q_EMPTY], kQTilesPerCta);
        for (int s2 = 0; s2 < kKStages; ++s2) {
            mbar_init(&bars[B_KRAW_FULL + s2], 1);
            mbar_init(&bars[B_K_FULL + s2], PAGED ? kRotThreads : 1);
            mbar_init(&bars[B_KPOS_FULL + s2], 32);
            mbar_init(&bars[B_K_EMPTY + s2], kQTilesPerCta);
            mbar_init(&bars[B_KPOS_FREE + s2], 256);
        }
        for (int s2 = 0; s2 < kVStages; ++s2) {
            mbar_init(&bars[B_VRAW_FULL + s2], 1);
            mbar_init(&bars[B_V_FULL + s2], PAGED ? 32 : 1);
            mbar_init(&bars[B_V_EMPTY + s2], kQTilesPerCta);
        }
        for (int t = 0; t < kQTilesPerCta; ++t) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&bars[B_S_FULL + 2 * t + b], 1);
                mbar_init(&bars[B_P_FULL + 2 * t + b], 128);
                mbar_init(&bars[B_PV_DONE + 2 * t + b], 1);
            }
            mbar_init(&bars[B_O_DONE + t], 1);
            mbar_init(&bars[B_O_FREE + t], 128);
        }
        for (int i = 0; i < 2 * kQTilesPerCta; ++i) mbar_init(&bars[B_DRAIN + i], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[B_ITEM_FULL + b], 1);
            mbar_init(&bars[B_ITEM_EMPTY + b], kItemReaders);
        }
        fence_mbar_init();
        misc[4] = 0;
        prefetch_tmap(&tm_q);
    }
    // up to here only the layout and shared memory were touched: the previous kernel (which
    // writes the rotated rows, the compacted keys and their positions) may still be running
    grid_dep_wait();
    grid_dep_launch();
    if (warp == kWarpMma) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), SM::kTmemCols);
        tmem_relinquish();
    }
    // (every K and V stage is filled whole: a cached tile by eight page copies, a page past the
    // request's last repeating that last page; a query-row tile by one copy whose rows past the
    // tensor's end read as 0; keys that are not there carry position kNoPos and are masked)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);

    // a reader's view of item `it`: false if the wait gave up
    auto take_item = [&](int it, AttnItem& w) -> bool {
        if (!mbar_wait(&bars[B_ITEM_FULL + (it & 1)], (it >> 1) & 1, abort_flag)) return false;
        w = slots[it & 1];
        return true;
    };

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ scheduler, Q and K producer
        if (lane == 0) {
            prefetch_tmap(&tm_kcache);
            if (!LSE) prefetch_tmap(&tm_kfresh);
        }
        const int Hkv = L[L_HKV];
        int kc = 0;                                   // K tiles this CTA issued before the item
        int last_k[kKStages] = {-1, -1}, last_q = -1;  // for the final drain
        bool ok = true;
        for (int it = 0; ok; ++it) {
            // the next item: the first is this CTA's own, the rest come in list order
            int idx = 0;
            if (lane == 0) idx = it == 0 ? (int)blockIdx.x : atomicAdd(prm.sched, 1) + (int)gridDim.x;
            idx = __shfl_sync(0xffffffffu, idx, 0);
            AttnItem w;
            w.req = -1;
            w.kvh = w.qpair = w.chunk = w.n_ct = w.n_ft = w.t0 = w.jb = w.n_loc = 0;
            w.n_rows = w.row_base = w.cbase = w.nsplit = w.slot_base = 0;
            w.lse_base = w.lse_chunks = 0;
            w.page_base = w.n_pages = w.n_sel = w.pad = 0;
            const int32_t* R = L;
            if (idx < n_items) {
                const int32_t* item = items + kItemWords * idx;
                w.req = item[0];
                w.kvh = item[1];
                w.qpair = item[2];
                w.chunk = item[3];
                R = L + L[L_OFF_REQ] + w.req * R_STRIDE;
                w.n_rows = LSE ? R[R_N_QUERY] : R[R_N_ROWS];
                w.row_base = R[R_ROW_BASE];
                w.cbase = R[R_CBASE];
                w.page_base = R[R_PAGE_BASE];
                w.n_pages = R[R_N_PAGES];
                w.n_sel = R[R_N_SEL];
                if (LSE) {
                    // LSE: tiles of all the request's cached tokens, cut into chunks
                    const int nkt = R[R_N_KTILES], chunks = R[R_LSE_CHUNKS];
                    const int tpc = (nkt + chunks - 1) / chunks;
                    w.t0 = w.chunk * tpc;
                    w.n_ct = max(0, min(tpc, nkt - w.t0));
                    w.n_loc = w.n_ct;
                    w.lse_base = R[R_LSE_BASE];
                    w.lse_chunks = chunks;
                } else {
                    // visible tiles: key positions increase along the cached tiles and along the
                    // fresh tiles, so each count is the number of tiles whose first key is at or
                    // before the pair's last row (the lanes test 32 tiles at a time).  Compacted:
                    // the cached tiles hold the kept cached keys and the fresh tiles every row of
                    // the request.  Paged: the cached tiles are the request's pool pages, a
                    // recomputed token's fresh key sitting in its cached copy's place, and only
                    // the query rows form fresh tiles.
                    const int n_rows_req = R[R_N_ROWS], n_sel = R[R_N_SEL];
                    const int32_t row_base = R[R_ROW_BASE];
                    const int row0 = w.qpair * kQTilesPerCta * toks_per_tile;
                    const int nrow = min(kQTilesPerCta * toks_per_tile, n_rows_req - row0);
                    const int32_t pmax = nrow > 0 ? prm.row_pos[row_base + row0 + nrow - 1] : -1;
                    int nct = 0, nft = 0;
                    if (PAGED) {
                        const int nkt = (R[R_N_PAGES] + kPagesPerTile - 1) / kPagesPerTile;
                        const int nft_total = (n_rows_req - n_sel + kTileKeys - 1) / kTileKeys;
                        const int32_t* pp = L + L[L_OFF_PAGEPOS] + R[R_PAGE_BASE];
                        for (int b = 0; b < nkt; b += 32)
                            nct += __popc(__ballot_sync(0xffffffffu, b + lane < nkt && pp[(b + lane) * kPagesPerTile] <= pmax));
                        for (int b = 0; b < nft_total; b += 32)
                            nft += __popc(__ballot_sync(0xffffffffu, b + lane < nft_total &&
                                                                         prm.row_pos[row_base + n_sel + (b + lane) * kTileKeys] <= pmax));
                    } else {
                        const int nkt = (R[R_N_PAGES] * kPage - n_sel + kTileKeys - 1) / kTileKeys;
                        const int nft_total = (n_rows_req + kTileKeys - 1) / kTileKeys;
                        const int32_t* kpc = prm.kpos_c + R[R_CBASE];
                        for (int b = 0; b < nkt; b += 32)
                            nct += __popc(__ballot_sync(0xffffffffu, b + lane < nkt && kpc[(b + lane) * kTileKeys] <= pmax));
                        for (int b = 0; b < nft_total; b += 32)
                            nft += __popc(__ballot_sync(0xffffffffu, b + lane < nft_total &&
                                                                         prm.row_pos[row_base + (b + lane) * kTileKeys] <= pmax));
                    }
                    const int32_t* PR = L + L[L_OFF_PAIR] + (R[R_PAIR_BASE] + w.qpair) * P_STRIDE;
                    const int n_all = nct + nft, ns = PR[P_NSPLIT];
                    w.n_ct = nct;
                    w.n_ft = nft;
                    w.nsplit = ns;
                    w.slot_base = PR[P_SLOT_BASE];
                    w.jb = (int)(((int64_t)w.chunk * n_all) / ns);
                    w.n_loc = (int)(((int64_t)(w.chunk + 1) * n_all) / ns) - w.jb;
                }
            }
            // publish it in slot it & 1 once every reader is done with item it - 2
            if (lane == 0) {
                ok = it < 2 || mbar_wait(&bars[B_ITEM_EMPTY + (it & 1)], ((it >> 1) - 1) & 1, abort_flag);
                if (ok) {
                    slots[it & 1] = w;
                    mbar_arrive(&bars[B_ITEM_FULL + (it & 1)]);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || w.req < 0) break;
            const int n_rows_req = LSE ? R[R_N_QUERY] : R[R_N_ROWS];
            const int32_t row_base = R[R_ROW_BASE];
            const int row0 = w.qpair * kQTilesPerCta * toks_per_tile;
            const int32_t kc_row0 = LSE ? w.kvh * L[L_TOTAL_TOKENS] + R[R_TOK_BASE] : 0;
            // first fresh row of the fresh tiles: paged, the request's first query row; compacted, its
            // first row
            const int32_t fbase = PAGED ? w.n_sel : 0;
            const int32_t kf_row0 = w.kvh * L[L_TOTAL_ROWS] + row_base + fbase;
            const int n_qrows = n_rows_req - fbase;
            const int n_kept = w.n_pages * kPage - w.n_sel;   // compacted cached keys of the request
            // key positions, which only the softmax waits for, and the pool rows of a cached tile's
            // pages: lane l holds the positions of keys 4l .. 4l+3 of a tile (kNoPos for a missing
            // key) and, for l < 8, the first pool row of page l of the tile (a page past the
            // request's last copies that last page instead: finite data whose keys are masked).
            // Loaded one tile ahead; the first tile's are requested now, before the Q buffer wait.
            const int n_ct = w.n_ct;
            const int32_t* page_pos = L + L[L_OFF_PAGEPOS] + w.page_base;
            const int32_t* blk = L + L[L_OFF_BLOCK] + w.page_base;
            // For a cached tile of the attention, lane l < 8 also loads page l's recompute bits and
            // the rank (among the request's recomputed tokens) of its first recomputed token.
            // It also loads 128 bytes of the tile's table rows: lane l takes 8 of the 32 float4 of
            // page l / 4 (the rows at the page's first position and, for d = 64, 8 positions on).
            auto meta = [&](int j, int32_t (&pos)[4], int32_t& prow, uint32_t& ex, int32_t& sel, float4 (&tr)[8]) {
                prow = 0;
                ex = 0u;
                sel = 0;
                if (j < n_ct && !LSE && !PAGED) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int ci = j * kTileKeys + 4 * lane + r;
                        pos[r] = ci < n_kept ? prm.kpos_c[w.cbase + ci] : kNoPos;
                    }
                } else if (j < n_ct) {
                    const int pg = (w.t0 + j) * kPagesPerTile;
                    const int lp = pg + lane / 4;   // keys 4l .. 4l+3 lie in page l / 4 of the tile
                    const int32_t p0 = lp < w.n_pages ? page_pos[lp] : kNoPos;
#pragma unroll
                    for (int r = 0; r < 4; ++r) pos[r] = lp < w.n_pages ? p0 + (4 * lane + r) % kPage : kNoPos;
                    if (PAGED) {
                        constexpr int F4 = D / 4;                 // float4 per table row
                        const int f0 = (lane % 4) * 8;            // this lane's first float4 of the page
                        const int32_t row = page_pos[lp < w.n_pages ? lp : w.n_pages - 1] + (f0 / F4) * (2 * D / 16);
                        const float4* src = reinterpret_cast<const float4*>(prm.rope + (int64_t)row * (D / 2)) + f0 % F4;
#pragma unroll
                        for (int q = 0; q < 8; ++q) tr[q] = src[q];
                    }
                    if (PAGED && lane < kPagesPerTile) {
                        prow = (blk[min(pg + lane, w.n_pages - 1)] * Hkv + w.kvh) * kPage;
                        if (!LSE && pg + lane < w.n_pages) {
                            ex = prm.excl[w.page_base + pg + lane];
                            sel = kPage * (pg + lane) - (prm.cidx[w.page_base + pg + lane] - w.cbase);
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int fr = (j - n_ct) * kTileKeys + 4 * lane + r;   // fresh row from fbase on
                        pos[r] = fr < n_qrows ? prm.row_pos[row_base + fbase + fr] : kNoPos;
                    }
                }
            };
            int32_t pos_n[4], prow_n = 0, sel_n = 0;
            uint32_t ex_n = 0;
            float4 tr_n[8];
            if (w.n_loc > 0) meta(w.jb, pos_n, prow_n, ex_n, sel_n, tr_n);
            // the item's Q tiles, once both Q K^T issuers are done with the previous item's
            if (lane == 0) {
                const int32_t qy = LSE ? (w.kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE] + row0) * g
                                       : (w.kvh * L[L_TOTAL_ROWS] + row_base + row0) * g;
                if (it > 0) {
                    // warm L2 with the Q rows while the previous item drains
                    for (int t = 0; t < kQTilesPerCta; ++t)
                        for (int hb = 0; hb < H; ++hb) tma_prefetch_2d(&tm_q, hb * 64, qy + t * kTileRows);
                    ok = mbar_wait(&bars[B_Q_EMPTY], (it - 1) & 1, abort_flag);
                }
                if (ok) {
                    mbar_arrive_expect_tx(&bars[B_Q_FULL], kQTilesPerCta * SM::kQ);
                    for (int t = 0; t < kQTilesPerCta; ++t)
                        for (int hb = 0; hb < H; ++hb)
                            tma_load_2d(sQ(t) + hb * 16384, &tm_q, &bars[B_Q_FULL], hb * 64, qy + t * kTileRows);
                    last_q = it;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            // its K tiles: the copies start as soon as the stage is free (the rotators wait only for
            // them); then the lanes write the tile's key positions
            for (int jj = 0; jj < w.n_loc; ++jj, ++kc) {
                const int j = w.jb + jj, ks = kc & 1;
                // paged: the copy lands on the rotators' barrier; otherwise the rotated copy is the
                // operand itself
                uint64_t* raw = &bars[(PAGED ? B_KRAW_FULL : B_K_FULL) + ks];
                const bool paged = PAGED && j < n_ct;
                // a cached tile holding recomputed tokens also brings their fresh keys: the block of
                // kStageRows fresh rows from the tile's first recomputed token on
                const bool stage_fresh = paged && __ballot_sync(0xffffffffu, lane < kPagesPerTile && ex_n != 0u) != 0u;
                const int32_t sel_first = __shfl_sync(0xffffffffu, sel_n, 0);
                if (lane == 0) {
                    ok = kc < kKStages || (mbar_wait(&bars[B_K_EMPTY + ks], ((kc >> 1) - 1) & 1, abort_flag) &&
                                           mbar_wait(&bars[B_KPOS_FREE + ks], ((kc >> 1) - 1) & 1, abort_flag));
                    if (ok) mbar_arrive_expect_tx(raw, H * 16384 + (stage_fresh ? SM::kKst : 0));
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (paged) {
                    // the tile's eight pool pages, 16 rows of this kv head each: lane 8*hb + m copies
                    // half hb of page m into its 2 KB slice of the stage
                    const int m = lane % kPagesPerTile, hb = lane / kPagesPerTile;
                    const int32_t y = __shfl_sync(0xffffffffu, prow_n, m);
                    if (lane < kPagesPerTile * H)
                        tma_load_2d(sKs(ks) + hb * 16384 + m * (kPage * 128), &tm_kcache, raw, hb * 64, y);
                    if (stage_fresh && lane == 0)
                        for (int hb2 = 0; hb2 < H; ++hb2)
                            tma_load_2d(sKst(ks) + hb2 * (kStageRows * 128), &tm_kstage, raw, hb2 * 64,
                                        w.kvh * L[L_TOTAL_ROWS] + row_base + sel_first);
                    if (lane < kPagesPerTile) sMeta(ks)[lane] = make_int2((int)ex_n, sel_n);
#pragma unroll
                    for (int q = 0; q < 8; ++q) sRope(ks)[lane * 8 + q] = tr_n[q];
                } else if (lane == 0) {
                    const CUtensorMap* map = j < n_ct ? &tm_kcache : &tm_kfresh;
                    const int32_t yc = LSE ? kc_row0 + (w.t0 + j) * kTileKeys
                                           : w.kvh * L[L_TOTAL_VALID] + w.cbase + j * kTileKeys;
                    const int32_t y = j < n_ct ? yc : kf_row0 + (j - n_ct) * kTileKeys;
                    for (int hb = 0; hb < H; ++hb) tma_load_2d(sKs(ks) + hb * 16384, map, raw, hb * 64, y);
                }
                last_k[ks] = kc;
                *reinterpret_cast<int4*>(sKpos(ks) + 4 * lane) = make_int4(pos_n[0], pos_n[1], pos_n[2], pos_n[3]);
                mbar_arrive(&bars[B_KPOS_FULL + ks]);
                if (jj + 1 < w.n_loc) meta(j + 1, pos_n, prow_n, ex_n, sel_n, tr_n);
            }
        }
        // every copy this warp started has landed before the CTA exits
        if (lane == 0) {
            if (last_q >= 0) mbar_drain(&bars[B_Q_FULL], last_q & 1);
            for (int s2 = 0; s2 < kKStages; ++s2)
                if (last_k[s2] >= 0) mbar_drain(&bars[(PAGED ? B_KRAW_FULL : B_K_FULL) + s2], (last_k[s2] >> 1) & 1);
        }
    } else if (warp == kWarpTmaV) {
        // ------------------------------------------------------------ V producer
        if (!LSE && !PAGED && lane == 0) {
            // compacted: the kept cached V rows (copied next to the compacted keys) or the fresh
            // rows, one copy per half of a tile
            prefetch_tmap(&tm_vcache);
            prefetch_tmap(&tm_vfresh);
            int vc = 0;
            int last_v[kVStages] = {-1, -1};
            for (int it = 0;; ++it) {
                AttnItem w;
                if (!take_item(it, w)) break;
                mbar_arrive(&bars[B_ITEM_EMPTY + (it & 1)]);
                if (w.req < 0) break;
                bool ok = true;
                for (int jj = 0; jj < w.n_loc; ++jj, ++vc) {
                    const int j = w.jb + jj, vs = vc & 1;
                    if (vc >= kVStages && !(ok = mbar_wait(&bars[B_V_EMPTY + vs], ((vc >> 1) - 1) & 1, abort_flag)))
                        break;
                    uint64_t* full = &bars[B_V_FULL + vs];
                    mbar_arrive_expect_tx(full, H * 16384);
                    if (j < w.n_ct) {
                        const int32_t y = w.kvh * L[L_TOTAL_VALID] + w.cbase + j * kTileKeys;
                        for (int hb = 0; hb < H; ++hb) tma_load_2d(sVs(vs) + hb * 16384, &tm_vcache, full, hb * 64, y);
                    } else {
                        const int32_t fr = w.row_base + (j - w.n_ct) * kTileKeys;
                        for (int hb = 0; hb < H; ++hb)
                            tma_load_3d(sVs(vs) + hb * 16384, &tm_vfresh, full, hb * 64, w.kvh, fr);
                    }
                    last_v[vs] = vc;
                }
                if (!ok) break;
            }
            for (int s2 = 0; s2 < kVStages; ++s2)
                if (last_v[s2] >= 0) mbar_drain(&bars[B_V_FULL + s2], (last_v[s2] >> 1) & 1);
        } else if (PAGED && !LSE) {
            // paged: V tiles of the cached pages (one copy per page and half, as for K) or of the
            // query rows.  Once a cached tile has landed, the recomputed tokens' cached V rows are
            // overwritten with their fresh rows: lane l takes page l / 4 of the tile and a quarter
            // of each row's 16-byte chunks.  The recompute bits are loaded one tile ahead and the
            // first fresh rows while the tile's copy is in flight.
            if (lane == 0) {
                prefetch_tmap(&tm_vcache);
                prefetch_tmap(&tm_vfresh);
            }
            const int Hkv = L[L_HKV];
            constexpr int CH = D / 8;          // 16-byte chunks per row
            constexpr int CPL = CH / 4;        // chunks per lane
            constexpr int kPre = 2;            // fresh rows loaded ahead per lane
            const int m = lane / 4, qtr = lane % 4;
            int vc = 0;
            int last_v[kVStages] = {-1, -1};
            auto stage_row = [&](int vs, int key, int ch) {
                return reinterpret_cast<uint4*>(sVs(vs) + (ch / 8) * 16384 + sw128_off(key, ch % 8));
            };
            bool ok = true;
            for (int it = 0; ok; ++it) {
                AttnItem w;
                ok = take_item(it, w);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_ITEM_EMPTY + (it & 1)]);
                if (w.req < 0) break;
                const int32_t* blk = L + L[L_OFF_BLOCK] + w.page_base;
                auto page_bits = [&](int j, uint32_t& ex, int& sel) {
                    ex = 0u;
                    sel = 0;
                    const int lp = j * kPagesPerTile + m;
                    if (j < w.n_ct && lp < w.n_pages) {
                        ex = prm.excl[w.page_base + lp];
                        if (ex) sel = kPage * lp - (prm.cidx[w.page_base + lp] - w.cbase);   // recomputed before it
                    }
                };
                uint32_t ex_n = 0;
                int sel_n = 0;
                if (w.n_loc > 0) page_bits(w.jb, ex_n, sel_n);
                for (int jj = 0; ok && jj < w.n_loc; ++jj, ++vc) {
                    const int j = w.jb + jj, vs = vc & 1;
                    uint64_t* raw = &bars[B_VRAW_FULL + vs];
                    if (lane == 0) {
                        ok = vc < kVStages || mbar_wait(&bars[B_V_EMPTY + vs], ((vc >> 1) - 1) & 1, abort_flag);
                        if (ok) mbar_arrive_expect_tx(raw, H * 16384);
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (j < w.n_ct) {
                        const int mm = lane % kPagesPerTile, hb = lane / kPagesPerTile;
                        if (lane < kPagesPerTile * H) {
                            const int lq = min(j * kPagesPerTile + mm, w.n_pages - 1);
                            tma_load_2d(sVs(vs) + hb * 16384 + mm * (kPage * 128), &tm_vcache, raw, hb * 64,
                                        (blk[lq] * Hkv + w.kvh) * kPage);
                        }
                    } else if (lane == 0) {
                        const int32_t fr = w.row_base + w.n_sel + (j - w.n_ct) * kTileKeys;
                        for (int hb = 0; hb < H; ++hb)
                            tma_load_3d(sVs(vs) + hb * 16384, &tm_vfresh, raw, hb * 64, w.kvh, fr);
                    }
                    last_v[vs] = vc;
                    uint32_t ex = ex_n;
                    int sel = sel_n;
                    // the first fresh rows, and the next tile's bits, while the copy is in flight
                    int pre_r[kPre], n_pre = 0;
                    uint4 pre[kPre][CPL];
#pragma unroll
                    for (int i = 0; i < kPre; ++i) {
                        if (ex != 0u && sel < w.n_sel) {
                            pre_r[i] = __ffs(ex) - 1;
                            const uint4* src = reinterpret_cast<const uint4*>(
                                prm.v_fresh + ((int64_t)(w.row_base + sel) * Hkv + w.kvh) * D);
#pragma unroll
                            for (int q = 0; q < CPL; ++q) pre[i][q] = src[qtr * CPL + q];
                            n_pre = i + 1;
                            ex &= ex - 1u;
                            ++sel;
                        }
                    }
                    if (jj + 1 < w.n_loc) page_bits(j + 1, ex_n, sel_n);
                    ok = mbar_wait(raw, (vc >> 1) & 1, abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
                    for (int i = 0; i < kPre; ++i)
                        if (i < n_pre)
#pragma unroll
                            for (int q = 0; q < CPL; ++q) *stage_row(vs, kPage * m + pre_r[i], qtr * CPL + q) = pre[i][q];
                    for (; ex != 0u; ex &= ex - 1u, ++sel) {   // rows beyond the first kPre
                        if (sel >= w.n_sel) { set_dev_error(kDevErrBounds); break; }
                        const int r = __ffs(ex) - 1;
                        const uint4* src = reinterpret_cast<const uint4*>(
                            prm.v_fresh + ((int64_t)(w.row_base + sel) * Hkv + w.kvh) * D);
                        uint4 v[CPL];
#pragma unroll
                        for (int q = 0; q < CPL; ++q) v[q] = src[qtr * CPL + q];
#pragma unroll
                        for (int q = 0; q < CPL; ++q) *stage_row(vs, kPage * m + r, qtr * CPL + q) = v[q];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    mbar_arrive(&bars[B_V_FULL + vs]);
                }
            }
            if (lane == 0)
                for (int s2 = 0; s2 < kVStages; ++s2)
                    if (last_v[s2] >= 0) mbar_drain(&bars[B_VRAW_FULL + s2], (last_v[s2] >> 1) & 1);
        }
    } else if (PAGED && warp >= kRot0 && warp < kRot0 + 2) {
        // ------------------------------------------------------------ K rotation (warps 14, 15)
        // MiniPIC 2.1: cached keys are rotated when used, to the request's logical positions.  A
        // cached tile holds 8 pool pages; thread t rotates 16-byte chunk pair c (dimensions 8c ..
        // 8c+7 and D/2 + 8c ..) of 2*CP consecutive keys of page m = t / 8, in place: bf16 in,
        // rotated fp16 out.  The keys of a page sit at consecutive positions p0 + r, so the
        // (cos, sin) pairs come from one table row (staged with the tile by the producer) and then
        // advance by one position step -- a rotation by theta_i, itself table row 1 -- from key to
        // key.  The arithmetic runs on packed fp32 pairs (two frequencies per instruction).  A
        // recomputed token's cached key is then overwritten with its fresh rotated key (same
        // position), which the producer staged with the tile as well.
        constexpr int CP = D / 16;
        constexpr int KPT = 2 * CP;
        const int rt = tid - kRot0 * 32;
        const int m = rt / 8, c = rt % CP, r0 = ((rt % 8) / CP) * KPT;
        const uint32_t o_hi = D == 128 ? 16384u : 0u;
        const int c_hi = D == 128 ? c : c + 4;
        const uint32_t st_hi = D == 128 ? (uint32_t)(kStageRows * 128) : 0u;
        const int f4 = m * 32 + (r0 / KPT) * (D / 4) + 4 * c;   // this thread's float4 in a staged table
        // one position step for frequencies 8c + 2e, 8c + 2e + 1: (cos, sin, -sin) as packed pairs
        uint64_t STC[4], STS[4], NSTS[4];
        {
            const float4* t1 = reinterpret_cast<const float4*>(prm.rope + D / 2 + 8 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 v = t1[e];
                STC[e] = f2_pack(v.x, v.z);
                STS[e] = f2_pack(v.y, v.w);
                NSTS[e] = f2_pack(-v.y, -v.w);
            }
        }
        int kc = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            AttnItem w;
            ok = take_item(it, w);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_ITEM_EMPTY + (it & 1)]);
            if (w.req < 0) break;
            for (int jj = 0; jj < w.n_loc; ++jj, ++kc) {
                const int j = w.jb + jj, ks = kc & 1;
                const bool rot = j < w.n_ct;
                ok = mbar_wait(&bars[B_KPOS_FULL + ks], (kc >> 1) & 1, abort_flag) &&
                     mbar_wait(&bars[B_KRAW_FULL + ks], (kc >> 1) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                if (rot) {
                    uint8_t* stage = sKs(ks);
                    // (cos, sin, -sin) at the first key, packed by frequency pairs
                    uint64_t C[4], S[4], NS[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 v = sRope(ks)[f4 + e];
                        C[e] = f2_pack(v.x, v.z);
                        S[e] = f2_pack(v.y, v.w);
                        NS[e] = f2_pack(-v.y, -v.w);
                    }
                    rotate_page_keys<D, KPT>(stage, kPage * m + r0, c, C, S, NS, STC, STS, NSTS);
                    // recomputed tokens: their fresh keys, already rotated to the same positions
                    const int2 pm = sMeta(ks)[m];
                    const int32_t sel_first = sMeta(ks)[0].y;
                    uint32_t ex = ((uint32_t)pm.x >> r0) & ((1u << KPT) - 1u);
                    int sel = pm.y + __popc((uint32_t)pm.x & ((1u << r0) - 1u));
                    for (; ex != 0u; ex &= ex - 1u, ++sel) {
                        const int key = kPage * m + r0 + __ffs(ex) - 1;
                        if (sel >= w.n_sel) { set_dev_error(kDevErrBounds); break; }
                        const int srow = sel - sel_first;
                        uint4 lo, hi;
                        if (srow < kStageRows) {
                            lo = *reinterpret_cast<const uint4*>(sKst(ks) + sw128_off(srow, c));
                            hi = *reinterpret_cast<const uint4*>(sKst(ks) + st_hi + sw128_off(srow, c_hi));
                        } else {   // beyond the staged block: from global memory
                            const __half* src = prm.k_rot + ((int64_t)w.kvh * L[L_TOTAL_ROWS] + w.row_base + sel) * D;
                            lo = *reinterpret_cast<const uint4*>(src + 8 * c);
                            hi = *reinterpret_cast<const uint4*>(src + D / 2 + 8 * c);
                        }
                        *reinterpret_cast<uint4*>(stage + sw128_off(key, c)) = lo;
                        *reinterpret_cast<uint4*>(stage + o_hi + sw128_off(key, c_hi)) = hi;
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(&bars[B_K_FULL + ks]);
            }
        }
    } else if (warp == kWarpMma || warp == kWarpMmaB || warp == kWarpPvA || warp == kWarpPvB) {
        // ------------------------------------------------------------ MMA issuers
        // The warp runs the loop converged (every lane waits, `ok` kept uniform by a vote) and
        // lane 0 alone issues: the descriptor arithmetic stays warp-uniform.
        const bool qk_role = warp == kWarpMma || warp == kWarpMmaB;
        const int t = (warp == kWarpMma || warp == kWarpPvA) ? 0 : 1;
        const uint32_t leader = lane == 0 ? 1u : 0u;
        if (qk_role || !LSE) {
            int hq = 0, kc = 0;   // halves / key tiles this CTA processed before the item
            bool ok = true;
            for (int it = 0; ok; ++it) {
                AttnItem w;
                ok = __all_sync(0xffffffffu, take_item(it, w));
                if (!ok) break;
                if (leader) mbar_arrive(&bars[B_ITEM_EMPTY + (it & 1)]);
                if (w.req < 0) break;
                const int nq = 2 * w.n_loc;   // halves of this item's key range
                if (qk_role && LSE) {
                    // LSE mode: Q K^T of a whole key tile (N = 128 keys: half the instructions of two
                    // halves) into S buffer kt & 1 of 128 columns, which the softmax frees once it has
                    // loaded the tile two before
                    constexpr uint32_t idesc_qk = idesc_f16(128, 128);
                    const uint32_t aQ = desc_sw128_lo(smem_u32(sQ(t)), 16);
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_Q_FULL], it & 1, abort_flag));
                    for (int j = 0; ok && j < w.n_loc; ++j) {
                        const int kt = kc + j;
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait(&bars[B_K_FULL + (kt & 1)], (kt >> 1) & 1, abort_flag) &&
                                            (kt < 2 || mbar_wait(&bars[B_P_FULL + 2 * t + (kt & 1)],
                                                                 ((kt - 2) >> 1) & 1, abort_flag)));
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t aK = desc_sw128_lo(smem_u32(sKs(kt & 1)), 16);
                        const uint32_t tS = tmem + t * 256 + (kt & 1) * 128;
#pragma unroll
                        for (int k4 = 0; k4 < D / 64; ++k4)   // 64 columns of d (one swizzle atom) a block
                            mma_ss_k4(leader, tS, aQ + k4 * 1024, aK + k4 * 1024, kDescSw128Hi, idesc_qk,
                                      k4 > 0 ? 1u : 0u);
                        mma_commit_by(leader, &bars[B_S_FULL + 2 * t + (kt & 1)]);
                        mma_commit_by(leader, &bars[B_K_EMPTY + (kt & 1)]);
                    }
                    if (ok) mma_commit_by(leader, &bars[B_Q_EMPTY]);
                } else if (qk_role) {
                    // Q K^T of half q = 2j + h of local key tile j: keys 64h .. 64h+63 into S buffer
                    // (hq + q) & 1, which the half two before it (P V done) frees
                    constexpr uint32_t idesc_qk = idesc_f16(128, 64);
                    const uint32_t aQ = desc_sw128_lo(smem_u32(sQ(t)), 16);
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_Q_FULL], it & 1, abort_flag));
                    for (int q = 0; ok && q < nq; ++q) {
                        const int hg = hq + q, kt = kc + (q >> 1), h = q & 1;
                        ok = __all_sync(0xffffffffu,
                                        (h == 1 || mbar_wait(&bars[B_K_FULL + (kt & 1)], (kt >> 1) & 1, abort_flag)) &&
                                            (hg < 2 || mbar_wait(&bars[B_PV_DONE + 2 * t + (hg & 1)],
                                                                 ((hg - 2) >> 1) & 1, abort_flag)));
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t aK = desc_sw128_lo(smem_u32(sKs(kt & 1)) + h * 64 * 128, 16);
                        const uint32_t tS = tmem + t * 128 + (hg & 1) * 64;
#pragma unroll
                        for (int k4 = 0; k4 < D / 64; ++k4)
                            mma_ss_k4(leader, tS, aQ + k4 * 1024, aK + k4 * 1024, kDescSw128Hi, idesc_qk,
                                      k4 > 0 ? 1u : 0u);
                        mma_commit_by(leader, &bars[B_S_FULL + 2 * t + (hg & 1)]);
                        if (h == 1) mma_commit_by(leader, &bars[B_K_EMPTY + (kt & 1)]);
                    }
                    if (ok) mma_commit_by(leader, &bars[B_Q_EMPTY]);
                } else {
                    // O += P(q) V(q): M=128, N=d in one instruction, K=64 keys in four steps; the
                    // item's first P V overwrites O once the softmax has read the previous item's
                    constexpr uint32_t idesc_pv = idesc_bf16(128, D, true);
                    const uint32_t tO = tmem + kTmemO + t * 128;
                    for (int q = 0; ok && q < nq; ++q) {
                        const int hg = hq + q, kt = kc + (q >> 1), h = q & 1;
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait(&bars[B_P_FULL + 2 * t + (hg & 1)], (hg >> 1) & 1, abort_flag) &&
                                            (h == 1 || mbar_wait(&bars[B_V_FULL + (kt & 1)], (kt >> 1) & 1, abort_flag)) &&
                                            (q > 0 || it == 0 ||
                                             mbar_wait(&bars[B_O_FREE + t], (it - 1) & 1, abort_flag)));
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t aV = desc_sw128_lo(smem_u32(sVs(kt & 1)) + h * 64 * 128, 16384);
                        const uint32_t tP = tmem + t * 128 + (hg & 1) * 64;
                        mma_ts_k4(leader, tO, tP, aV, kDescSw128Hi, idesc_pv, q > 0 ? 1u : 0u);
                        mma_commit_by(leader, &bars[B_PV_DONE + 2 * t + (hg & 1)]);
                        if (h == 1) mma_commit_by(leader, &bars[B_V_EMPTY + (kt & 1)]);
                    }
                    if (ok) mma_commit_by(leader, &bars[B_O_DONE + t]);
                }
                hq += nq;
                kc += w.n_loc;
            }
            const int di = (qk_role ? 0 : 2) + t;
            mma_commit_by(leader, &bars[B_DRAIN + di]);
            if (leader) mbar_drain(&bars[B_DRAIN + di], 0);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-7)
        // Group t (warps 4t..4t+3) owns Q tile t.  Scores arrive already in log2 units: the
        // rotated query rows carry log2(e)/sqrt(d).
        const int t = warp >= kWarpSoftB ? 1 : 0;
        const int m = tid - t * 128;           // tile row = TMEM lane
        const int tok = m / g, hl = m % g;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tO = tmem + lane_addr + kTmemO + t * 128;
        int hq = 0, kc = 0;   // halves / key tiles this CTA processed before the item
        bool ok = true;
        bool have_pre = false;   // this row's position for the item was loaded during the last epilogue
        int32_t pos_pre = -1;
        for (int it = 0; ok; ++it) {
            AttnItem w;
            ok = take_item(it, w);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_ITEM_EMPTY + (it & 1)]);
            if (w.req < 0) break;
            const int n_rows_req = w.n_rows;
            const int32_t row_base = w.row_base;
            const int row = w.qpair * kQTilesPerCta * toks_per_tile + t * toks_per_tile + tok;
            const bool valid = row < n_rows_req;
            int32_t mypos;
            if (LSE) mypos = valid ? kNoPos - 1 : -1;
            else mypos = have_pre ? pos_pre : (valid ? prm.row_pos[row_base + row] : -1);
            have_pre = false;
            // output locations, fixed before the tile loop so that only one pointer stays live
            // across it (a split key range writes a normalized partial row plus its max and sum)
            __nv_bfloat16* out_row = nullptr;
            float2* ml_slot = nullptr;
            if (valid) {
                if (LSE) {
                    // [kv head][chunk][query row]: a warp's 32 rows are contiguous
                    ml_slot = prm.lse_part + w.lse_base +
                              ((int64_t)w.kvh * w.lse_chunks + w.chunk) * (n_rows_req * g) + row * g + hl;
                } else {
                    if (w.nsplit == 1) {
                        out_row = prm.out + ((int64_t)(row_base + row) * Hq + w.kvh * g + hl) * D;
                    } else {
                        const int64_t prow = (int64_t)(w.slot_base + w.kvh * w.nsplit + w.chunk) *
                                                 (kQTilesPerCta * kTileRows) + t * kTileRows + m;
                        out_row = prm.part_o + prow * D;
                        ml_slot = prm.part_ml + prow;
                    }
                }
            }
            if (PAGED && !LSE) {   // parked in shared memory across the tile loop, where registers are scarce
                volatile uint64_t* park = reinterpret_cast<volatile uint64_t*>(smem + SM::oPark) + 2 * (warp * 32 + lane);
                park[0] = reinterpret_cast<uint64_t>(out_row);
                park[1] = reinterpret_cast<uint64_t>(ml_slot);
            }
            float m_run = -INFINITY, l_run = 0.f;
            int cut = 0;
            const int nq = 2 * w.n_loc;
            if constexpr (LSE) {
                // LSE mode: S of a whole key tile per buffer (128 columns), read in two 64-column
                // parts; the buffer is released once both parts are in registers (nothing goes
                // back to TMEM), the running max and sum are kept as in the attention
                for (int j = 0; j < w.n_loc; ++j) {
                    const int kt = kc + j, ks = kt & 1;
                    const uint32_t tS0 = tmem + lane_addr + t * 256 + ks * 128;
                    ok = mbar_wait(&bars[B_S_FULL + 2 * t + ks], (kt >> 1) & 1, abort_flag) &&
                         mbar_wait(&bars[B_KPOS_FULL + ks], (kt >> 1) & 1, abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    {
                        // visible keys of this row: a prefix of the tile (missing keys carry kNoPos)
                        const int32_t* kp = sKpos(ks);
                        if (kp[kTileKeys - 1] <= mypos) {
                            cut = kTileKeys;
                        } else {
                            int lo = 0;
#pragma unroll
                            for (int step = 64; step >= 1; step >>= 1)
                                if (kp[lo + step - 1] <= mypos) lo += step;
                            cut = lo;
                        }
                        mbar_arrive(&bars[B_KPOS_FREE + ks]);
                    }
                    if constexpr (!PAGED) {
                        // the whole key tile's 128 scores in registers (12 warps leave room), the S
                        // buffer released as soon as they have landed
                        const bool full = __all_sync(0xffffffffu, cut >= kTileKeys);
                        uint32_t sv[128];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
                            tmem_ld32(tS0 + c4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c4 * 32]));
                        tmem_ld_wait();
                        tc_fence_before();
                        mbar_arrive(&bars[B_P_FULL + 2 * t + ks]);
                        if (!full) {
#pragma unroll
                            for (int e = 0; e < 128; ++e)
                                if (e >= cut) sv[e] = __float_as_uint(-INFINITY);
                        }
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int e = 0; e < 128; e += 8) {
                            m4[0] = max3f(m4[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                            m4[1] = max3f(m4[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                            m4[2] = max3f(m4[2], __uint_as_float(sv[e + 4]), __uint_as_float(sv[e + 5]));
                            m4[3] = max3f(m4[3], __uint_as_float(sv[e + 6]), __uint_as_float(sv[e + 7]));
                        }
                        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                        const float m_new = fmaxf(m_run, mx);
                        if (m_new > m_run + 8.0f) {   // lazy rescale: keep the terms <= 2^8
                            l_run *= ex2(m_run - m_new);
                            m_run = m_new;
                        }
                        const float msub = m_run == -INFINITY ? 0.f : m_run;
                        const uint64_t negm2 = f2_pack(-msub, -msub);
                        uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                        for (int e = 0; e < 64; ++e) {
                            float d0, d1;
                            f2_unpack(f2_add(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), negm2), d0, d1);
                            acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(ex2(d0), ex2(d1)));
                        }
                        float a0, a1, b0, b1;
                        f2_unpack(acc2[0], a0, a1);
                        f2_unpack(acc2[1], b0, b1);
                        l_run += (a0 + b0) + (a1 + b1);
                    } else
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const int cut_h = cut - 64 * h;
                        const bool full = __all_sync(0xffffffffu, cut_h >= 64);
                        uint32_t sv[64];
                        tmem_ld32(tS0 + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                        tmem_ld32(tS0 + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                        tmem_ld_wait();
                        if (h == 1) {
                            tc_fence_before();
                            mbar_arrive(&bars[B_P_FULL + 2 * t + ks]);
                        }
                        if (!full) {
#pragma unroll
                            for (int e = 0; e < 64; ++e)
                                if (e >= cut_h) sv[e] = __float_as_uint(-INFINITY);
                        }
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int e = 0; e < 64; e += 8) {
                            m4[0] = max3f(m4[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                            m4[1] = max3f(m4[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                            m4[2] = max3f(m4[2], __uint_as_float(sv[e + 4]), __uint_as_float(sv[e + 5]));
                            m4[3] = max3f(m4[3], __uint_as_float(sv[e + 6]), __uint_as_float(sv[e + 7]));
                        }
                        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                        const float m_new = fmaxf(m_run, mx);
                        if (m_new > m_run + 8.0f) {   // lazy rescale: keep the terms <= 2^8
                            l_run *= ex2(m_run - m_new);
                            m_run = m_new;
                        }
                        const float msub = m_run == -INFINITY ? 0.f : m_run;
                        const uint64_t negm2 = f2_pack(-msub, -msub);
                        uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float d0, d1;
                            f2_unpack(f2_add(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), negm2), d0, d1);
                            acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(ex2(d0), ex2(d1)));
                        }
                        float a0, a1, b0, b1;
                        f2_unpack(acc2[0], a0, a1);
                        f2_unpack(acc2[1], b0, b1);
                        l_run += (a0 + b0) + (a1 + b1);
                    }
                }
            } else
            for (int q = 0; q < nq; ++q) {    // halves of the item's key tiles
                const int hg = hq + q, kt = kc + (q >> 1), h = q & 1, ks = kt & 1;
                const uint32_t tS = tmem + lane_addr + t * 128 + (hg & 1) * 64;
                ok = mbar_wait(&bars[B_S_FULL + 2 * t + (hg & 1)], (hg >> 1) & 1, abort_flag);
                if (h == 0) ok = ok && mbar_wait(&bars[B_KPOS_FULL + ks], (kt >> 1) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                if (h == 0) {
                    // causal limit of this row inside the tile: keys are in increasing position
                    // order, so the visible ones are a prefix (binary search)
                    const int32_t* kp = sKpos(ks);
                    if (kp[kTileKeys - 1] <= mypos) {
                        cut = kTileKeys;         // the whole tile is visible (the common case)
                    } else {
                        int lo = 0;
#pragma unroll
                        for (int step = 64; step >= 1; step >>= 1)
                            if (kp[lo + step - 1] <= mypos) lo += step;
                        cut = lo;                // <= 127: key 127 is not visible
                    }
                    mbar_arrive(&bars[B_KPOS_FREE + ks]);
                }
                const int cut_h = cut - 64 * h;   // visible keys of this half: [0, cut_h)
                const bool full = __all_sync(0xffffffffu, cut_h >= 64);
                // the half's 64 scores in registers (one wait for both loads)
                uint32_t sv[64];
                tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                tmem_ld_wait();
                if (!full) {
                    // keys at or beyond the causal limit leave the row: score -inf
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (e >= cut_h) sv[e] = __float_as_uint(-INFINITY);
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 64; e += 8) {
                    m4[0] = max3f(m4[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    m4[1] = max3f(m4[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                    m4[2] = max3f(m4[2], __uint_as_float(sv[e + 4]), __uint_as_float(sv[e + 5]));
                    m4[3] = max3f(m4[3], __uint_as_float(sv[e + 6]), __uint_as_float(sv[e + 7]));
                }
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                const float m_new = fmaxf(m_run, mx);
                const bool need = m_new > m_run + 8.0f;     // lazy rescale: keep P <= 2^8
                const float alpha = need ? ex2(m_run - m_new) : 1.0f;
                if (need) { l_run *= alpha; m_run = m_new; }
                const float msub = m_run == -INFINITY ? 0.f : m_run;
                // p = 2^(s - m); P (bf16 pairs) goes over the half's first 32 S columns.  The
                // subtraction and the running sums use packed fp32 pairs.
                const uint64_t negm2 = f2_pack(-msub, -msub);
                uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float d0, d1;
                    f2_unpack(f2_add(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), negm2), d0, d1);
                    const float p0 = ex2(d0), p1 = ex2(d1);
                    acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(p0, p1));
                    pk[e] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tS, pk);
                {
                    float a0, a1, b0, b1;
                    f2_unpack(acc2[0], a0, a1);
                    f2_unpack(acc2[1], b0, b1);
                    l_run += (a0 + b0) + (a1 + b1);
                }
                {
                    if (q > 0 && __any_sync(0xffffffffu, need)) {
                        // every earlier P V of this tile must be done before O is rescaled
                        ok = mbar_wait(&bars[B_PV_DONE + 2 * t + ((hg - 1) & 1)], ((hg - 1) >> 1) & 1, abort_flag);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < D / 32; ++cc) {
                            uint32_t o[32];
                            tmem_ld32(tO + cc * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + cc * 32, o);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bars[B_P_FULL + 2 * t + (hg & 1)]);
                }
            }
            if (!ok) break;
            if (PAGED && !LSE) {
                volatile uint64_t* park = reinterpret_cast<volatile uint64_t*>(smem + SM::oPark) + 2 * (warp * 32 + lane);
                out_row = reinterpret_cast<__nv_bfloat16*>(park[0]);
                ml_slot = reinterpret_cast<float2*>(park[1]);
            }
            if (ml_slot != nullptr) *ml_slot = make_float2(w.n_loc > 0 ? m_run : -INFINITY, l_run);
            if (!LSE) {
                // if the next item is already published, start loading this row's position for it
                // now, so that the load runs under the epilogue
                if (__all_sync(0xffffffffu, mbar_test_wait(&bars[B_ITEM_FULL + ((it + 1) & 1)], ((it + 1) >> 1) & 1))) {
                    const AttnItem& wn = slots[(it + 1) & 1];
                    if (wn.req >= 0) {
                        const int rn = wn.qpair * kQTilesPerCta * toks_per_tile + t * toks_per_tile + tok;
                        pos_pre = rn < wn.n_rows ? prm.row_pos[wn.row_base + rn] : -1;
                        have_pre = true;
                    }
                }
                // epilogue: O / l once the item's last P V is done (an item without key tiles has no
                // O to read); then O is free for the next item's first P V
                ok = mbar_wait(&bars[B_O_DONE + t], it & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                if (w.n_loc > 0) {
                    const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_ld_wait();
                        if (out_row != nullptr) {
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                uint4 v;
                                v.x = pack_bf16x2(__uint_as_float(o[8 * qq + 0]) * inv, __uint_as_float(o[8 * qq + 1]) * inv);
                                v.y = pack_bf16x2(__uint_as_float(o[8 * qq + 2]) * inv, __uint_as_float(o[8 * qq + 3]) * inv);
                                v.z = pack_bf16x2(__uint_as_float(o[8 * qq + 4]) * inv, __uint_as_float(o[8 * qq + 5]) * inv);
                                v.w = pack_bf16x2(__uint_as_float(o[8 * qq + 6]) * inv, __uint_as_float(o[8 * qq + 7]) * inv);
                                *reinterpret_cast<uint4*>(out_row + cc * 32 + 8 * qq) = v;
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars[B_O_FREE + t]);
            }
            hq += nq;
            kc += w.n_loc;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, SM::kTmemCols);
    }
}

}  // namespace pcf
