// Flash-style attention over the position-free paged cache with in-kernel RoPE (sm_103a).
//
// MiniPIC, section 2.1: cached keys k~_j stay unrotated in shared pages; the attention kernel
// rotates them on the fly to the key's per-request logical position pi(j) with a cos/sin lookup
// and fused multiply-adds, so score(t, j) = (R_t q_t)^T (R_pi(j) k~_j) / sqrt(d).
// QCFuse, section 2C / Phase 4 (and the sparse attention kernel of its section 3): the recomputed
// tokens and the query tokens attend over the cached keys minus the recomputed ones plus the
// fresh rows, keeping causal order on logical positions.
//
// One CTA = two tiles A and B of 128 query rows each (a tile packs the g query heads of 128/g
// consecutive rows of one request, all sharing kv head `kvh`) against the request's KV tiles of
// 128 keys; both tiles share every rotated K tile and every V tile:
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: S row from TMEM, mask, online
//               softmax (lazy rescale), P -> TMEM (over the S columns), O epilogue
//   warps 8-11  rotate cached K tiles in shared memory (in place, 128-byte swizzled K-major)
//   warp  12    TMEM allocation + single-thread tcgen05.mma issue, in the order
//               PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1), so that the tensor core works on one tile
//               while the other tile's softmax runs
//   warp  13    K producer (TMA): Q tiles, cached K pages through the block table with their page
//               cos/sin rows, fresh K tiles; 2-stage ring, freed by the second QK^T of a stage
//   warp  14    V producer (TMA): cached V pages / fresh V tiles; 2-stage ring, freed by PV_B
// TMEM: S_A / P_A at columns [0,128), S_B / P_B at [128,256), O_A at [256,256+d), O_B at
// [384,384+d).  S = Q K^T is fp16 x fp16 (M=128, N=128 keys, K=d); P (bf16) overwrites its own S
// columns and is the A operand of O += P V (M=128, N=d, V as an MN-major bf16 operand).
// Keys that do not take part (recomputed tokens' cached copies, missing pages or rows) are
// removed by the tensor core itself: Q K^T gets one more K=16 step whose A slab is a column of
// ones and whose B slab carries 0 or -30000 per key, so their scores (log2 units) underflow to
// P = 0; only rows whose causal limit falls inside a tile need per-element masking.
// LSE mode (critical-layer scoring, pass 1) runs the same pipeline without P/V and writes the
// per-row running max and sum of one key chunk.
#pragma once
#include "layout_format.h"
#include "ptx.cuh"

namespace pcf {

constexpr int kAttnThreads = 480;   // 15 warps
constexpr int kWarpSoftB = 4;
constexpr int kWarpRot0 = 8;
constexpr int kWarpMma = 12;
constexpr int kWarpTma = 13;
constexpr int kWarpTmaV = 14;
constexpr int kNoPos = 0x7FFFFFFF;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kTmemO = 256;     // O_A at 256, O_B at 384
constexpr int kSlab16 = kTileRows * 16 * 2;   // one [128][16] fp16 bias slab
constexpr float kKeyOff = -30000.f;           // bias of a key that does not take part

struct AttnParams {
    const int32_t* layout;
    const uint16_t* excl;      // attention: per logical page exclusion bits
    const int32_t* row_pos;    // attention: logical position of every row
    const float2* rope;        // [max_pos][D/2] (cos, sin)
    __nv_bfloat16* out;        // attention: [rows][Hq][D]
    float2* lse_part;          // LSE: (running max in log2 units, running sum) per row and chunk
    __nv_bfloat16* part_o;     // attention with a split key range: normalized partial O per slot
    float2* part_ml;           //   and its (running max, running sum) per row
};

template <int D, bool LSE>
struct AttnSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kQ = kTileRows * D * 2;          // one Q tile
    static constexpr int kK = kTileKeys * D * 2;
    static constexpr int kV = LSE ? 0 : kTileKeys * D * 2;
    static constexpr int kCs = kPagesPerTile * (D / 2) * 8;
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kQTilesPerCta * kQ;
    static constexpr int oV = oK + kKStages * kK;
    static constexpr int oCs = oV + kVStages * kV;
    static constexpr int oKpos = oCs + kKStages * kCs;
    static constexpr int oQaug = oKpos + kKStages * kTileKeys * 4;   // ones column (1024-aligned)
    static constexpr int oKaug = oQaug + kSlab16;                    // per K stage: key bias column
    static constexpr int oBar = oKaug + kKStages * kSlab16;
    static constexpr int kNumBars = 24;
    static constexpr int oMisc = oBar + kNumBars * 8;
    static constexpr int kBytes = oMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;   // slack for 1024-byte alignment
    static constexpr uint32_t kTmemCols = LSE ? 256 : 512;
};

// barrier slots
enum : int {
    B_Q_FULL = 0,
    B_K_FULL = 1,      // [2] K pages (+ cos/sin rows) landed
    B_KROT_FULL = 3,   // [2] K tile rotated, key positions and validity written
    B_K_EMPTY = 5,     // [2] both Q K^T that read the stage are done
    B_KPOS_FREE = 7,   // [2] both softmax groups are done with the stage's key info (256 arrivals)
    B_V_FULL = 9,      // [2]
    B_V_EMPTY = 11,    // [2] P_B V that read the stage is done
    B_S_FULL = 13,     // [2] per Q tile: S = Q K^T landed
    B_S_FREE = 15,     // [2] per Q tile (LSE mode): softmax done reading S
    B_P_FULL = 17,     // [2] per Q tile: P written, O rescaled
    B_PV_DONE = 19,    // [2] per Q tile: P V done (O final for this tile, S/P columns free)
    B_DRAIN = 21
};

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.y, b.x, a.x * b.y));
}

// Rotate the 8 pairs (i, i + D/2), i = 8c .. 8c+7, of key row `row` in a swizzled K tile, in place:
// bf16 in (the unrotated page), fp16 out (operand of the fp16 Q K^T).
template <int D>
__device__ __forceinline__ void rotate_chunk_pair(uint8_t* sK, int row, int c, const float2 (&cs)[8]) {
    uint8_t* pa;
    uint8_t* pb;
    if (D == 128) {
        pa = sK + sw128_off(row, c);
        pb = sK + 16384 + sw128_off(row, c);
    } else {
        pa = sK + sw128_off(row, c);
        pb = sK + sw128_off(row, c + 4);
    }
    const uint4 a = *reinterpret_cast<const uint4*>(pa);
    const uint4 b = *reinterpret_cast<const uint4*>(pb);
    const uint32_t ia[4] = {a.x, a.y, a.z, a.w};
    const uint32_t ib[4] = {b.x, b.y, b.z, b.w};
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 c0 = cs[2 * e], c1 = cs[2 * e + 1];
        const float a0 = bf16_lo(ia[e]), a1 = bf16_hi(ia[e]);
        const float b0 = bf16_lo(ib[e]), b1 = bf16_hi(ib[e]);
        oa[e] = pack_f16x2(fmaf(a0, c0.x, -b0 * c0.y), fmaf(a1, c1.x, -b1 * c1.y));
        ob[e] = pack_f16x2(fmaf(b0, c0.x, a0 * c0.y), fmaf(b1, c1.x, a1 * c1.y));
    }
    *reinterpret_cast<uint4*>(pa) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4*>(pb) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// Rotation of one cached K tile by 128 threads (rt = 0..127).  Thread (c, pg, rg) owns chunk pair
// c of rows rg*RPT .. rg*RPT+RPT-1 of page pg; it composes the page-base angle (table row of the
// page's first position, in sCs) with its first row's offset once and then advances the angle by
// one position per row.  All rows are loaded before any is stored (no shared-memory round trip
// per row).  Rows of missing pages hold stale finite data and are masked by the softmax.
template <int D>
__device__ __forceinline__ int rot_page_of(int rt) { return (rt / (D / 16)) % kPagesPerTile; }

template <int D>
__device__ __forceinline__ void rotate_cached_tile(uint8_t* sK, const float2* sCs, int rt,
                                                   const float2* __restrict__ cs_start_g, const float2 (&cs_step)[8]) {
    constexpr int CPR = D / 16;
    constexpr int RGN = kTileKeys / (CPR * kPagesPerTile);
    constexpr int RPT = kPage / RGN;
    const int c = rt % CPR;
    const int pg = (rt / CPR) % kPagesPerTile;
    const int rg = rt / (CPR * kPagesPerTile);
    const int row0 = pg * kPage + rg * RPT;
    uint8_t* base_a = sK;
    uint8_t* base_b = sK + (D == 128 ? 16384 : 0);
    const int cb = D == 128 ? c : c + 4;
    float2 cs[8];
    const float4* b4 = reinterpret_cast<const float4*>(sCs + pg * (D / 2) + 8 * c);
    const float4* s4 = reinterpret_cast<const float4*>(cs_start_g);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 v = b4[q];
        const float4 w = __ldg(s4 + q);
        cs[2 * q] = cmul(make_float2(v.x, v.y), make_float2(w.x, w.y));
        cs[2 * q + 1] = cmul(make_float2(v.z, v.w), make_float2(w.z, w.w));
    }
    // rows are independent: the next row is loaded before the current one is written back
    uint4 a_nx = *reinterpret_cast<const uint4*>(base_a + sw128_off(row0, c));
    uint4 b_nx = *reinterpret_cast<const uint4*>(base_b + sw128_off(row0, cb));
#pragma unroll 1
    for (int r = 0; r < RPT; ++r) {
        const uint4 a = a_nx, b = b_nx;
        if (r + 1 < RPT) {
            a_nx = *reinterpret_cast<const uint4*>(base_a + sw128_off(row0 + r + 1, c));
            b_nx = *reinterpret_cast<const uint4*>(base_b + sw128_off(row0 + r + 1, cb));
        }
        const uint32_t ia[4] = {a.x, a.y, a.z, a.w};
        const uint32_t ib[4] = {b.x, b.y, b.z, b.w};
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 c0 = cs[2 * e], c1 = cs[2 * e + 1];
            const float a0 = bf16_lo(ia[e]), a1 = bf16_hi(ia[e]);
            const float b0 = bf16_lo(ib[e]), b1 = bf16_hi(ib[e]);
            oa[e] = pack_f16x2(fmaf(a0, c0.x, -b0 * c0.y), fmaf(a1, c1.x, -b1 * c1.y));
            ob[e] = pack_f16x2(fmaf(b0, c0.x, a0 * c0.y), fmaf(b1, c1.x, a1 * c1.y));
        }
        *reinterpret_cast<uint4*>(base_a + sw128_off(row0 + r, c)) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
        *reinterpret_cast<uint4*>(base_b + sw128_off(row0 + r, cb)) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
#pragma unroll
        for (int i = 0; i < 8; ++i) cs[i] = cmul(cs[i], cs_step[i]);
    }
}

// 15 warps: 4 per SM sub-partition at most, so each thread may hold up to 128 registers; the
// softmax works on 32-key slices of the S row to stay below that.
template <int D, bool LSE>
__global__ void __launch_bounds__(kAttnThreads)
attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kpool,
            const __grid_constant__ CUtensorMap tm_vpool, const __grid_constant__ CUtensorMap tm_kfresh,
            const __grid_constant__ CUtensorMap tm_vfresh, const AttnParams prm) {
    using SM = AttnSmem<D, LSE>;
    constexpr int H = SM::kHalves;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sQ = [&](int t) { return smem + SM::oQ + t * SM::kQ; };
    auto sKs = [&](int st) { return smem + SM::oK + st * SM::kK; };
    auto sVs = [&](int st) { return smem + SM::oV + st * SM::kV; };
    auto sCs = [&](int st) { return reinterpret_cast<float2*>(smem + SM::oCs + st * SM::kCs); };
    auto sKpos = [&](int st) { return reinterpret_cast<int32_t*>(smem + SM::oKpos) + st * kTileKeys; };
    uint8_t* sQaug = smem + SM::oQaug;
    auto sKaug = [&](int st) { return smem + SM::oKaug + st * kSlab16; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::oBar);
    int32_t* misc = reinterpret_cast<int32_t*>(smem + SM::oMisc);
    // misc: [0] tmem base, [1] n cached tiles, [2] n fresh tiles, [3] first cached tile, [4] abort,
    //       [5] first tile of this CTA's key range, [6] end of the range (tiles in visible order)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* L = prm.layout;
    const int32_t* item = L + (LSE ? L[L_OFF_LSE] : L[L_OFF_ATTN]) + kItemWords * blockIdx.x;
    const int req = item[0], kvh = item[1], qpair = item[2], chunk = item[3];   // chunk: LSE key chunk
                                                                                  // or attention split
    const int32_t* R = L + L[L_OFF_REQ] + req * R_STRIDE;
    const int Hq = L[L_HQ], Hkv = L[L_HKV], g = L[L_GROUP];
    const int toks_per_tile = kTileRows / g;
    const int n_rows_req = LSE ? R[R_N_QUERY] : R[R_N_ROWS];
    const int row0 = qpair * kQTilesPerCta * toks_per_tile;        // first row of tile A
    const int nrow_cta = min(kQTilesPerCta * toks_per_tile, n_rows_req - row0);
    const int n_pages = R[R_N_PAGES];
    const int32_t page_base = R[R_PAGE_BASE];
    const int32_t row_base = R[R_ROW_BASE];
    const int32_t* page_pos = L + L[L_OFF_PAGEPOS] + page_base;
    const int32_t* blk = L + L[L_OFF_BLOCK] + page_base;

    if (tid == 0) {
        mbar_init(&bars[B_Q_FULL], 1);
        for (int s2 = 0; s2 < kKStages; ++s2) {
            mbar_init(&bars[B_K_FULL + s2], 1);
            mbar_init(&bars[B_KROT_FULL + s2], 128);
            mbar_init(&bars[B_K_EMPTY + s2], 1);
            mbar_init(&bars[B_KPOS_FREE + s2], 256);
        }
        for (int s2 = 0; s2 < kVStages; ++s2) {
            mbar_init(&bars[B_V_FULL + s2], 1);
            mbar_init(&bars[B_V_EMPTY + s2], 1);
        }
        for (int t = 0; t < kQTilesPerCta; ++t) {
            mbar_init(&bars[B_S_FULL + t], 1);
            mbar_init(&bars[B_S_FREE + t], 128);
            mbar_init(&bars[B_P_FULL + t], 128);
            mbar_init(&bars[B_PV_DONE + t], 1);
        }
        mbar_init(&bars[B_DRAIN], 1);
        fence_mbar_init();
        int nct, nft = 0, t0 = 0;
        const int nkt = R[R_N_KTILES];
        if (LSE) {
            const int chunks = R[R_LSE_CHUNKS];
            const int tpc = (nkt + chunks - 1) / chunks;
            t0 = chunk * tpc;
            nct = max(0, min(tpc, nkt - t0));
        } else {
            const int32_t pmax = nrow_cta > 0 ? prm.row_pos[row_base + row0 + nrow_cta - 1] : -1;
            nct = 0;
            while (nct < nkt && page_pos[nct * kPagesPerTile] <= pmax) ++nct;
            const int nft_total = (n_rows_req + kTileKeys - 1) / kTileKeys;
            while (nft < nft_total && prm.row_pos[row_base + nft * kTileKeys] <= pmax) ++nft;
        }
        misc[1] = nct;
        misc[2] = nft;
        misc[3] = t0;
        misc[4] = 0;
        const int n_all = nct + nft;
        const int ns = LSE ? 1 : R[R_NSPLIT];
        const int sp = LSE ? 0 : chunk;
        misc[5] = (int)(((int64_t)sp * n_all) / ns);
        misc[6] = (int)(((int64_t)(sp + 1) * n_all) / ns);
    }
    if (warp == kWarpMma) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), SM::kTmemCols);
        tmem_relinquish();
    }
    // V stages start finite (keys masked to P = 0 then contribute 0 * V); bias slabs start at 0
    // with a column of ones on the query side
    if (!LSE) {
        uint4* z = reinterpret_cast<uint4*>(smem + SM::oV);
        for (int i = tid; i < (kVStages * SM::kV) / 16; i += kAttnThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
    {
        uint4* z = reinterpret_cast<uint4*>(sQaug);
        for (int i = tid; i < ((1 + kKStages) * kSlab16) / 16; i += kAttnThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (tid < kTileRows) *reinterpret_cast<__half*>(sQaug + slab16_off(tid, 0)) = __float2half(1.0f);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);
    const int n_ct = misc[1], n_ft = misc[2], t0 = misc[3];
    const int n_tiles = n_ct + n_ft;
    const int jb = misc[5], n_loc = misc[6] - misc[5];   // tiles jb .. jb+n_loc-1 of the visible range
    const int n_phys = L[L_N_PHYS];

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ K producer
        // Lane p (< 8) fetches the block-table entry and position of page p of the next tile while
        // the current tile is issued, then issues that page's copies itself.
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_kpool);
            if (!LSE) prefetch_tmap(&tm_kfresh);
            const int32_t qy = LSE ? (kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE] + row0) * g
                                   : (kvh * L[L_TOTAL_ROWS] + row_base + row0) * g;
            mbar_arrive_expect_tx(&bars[B_Q_FULL], kQTilesPerCta * SM::kQ);
            for (int t = 0; t < kQTilesPerCta; ++t)
                for (int hb = 0; hb < H; ++hb)
                    tma_load_2d(sQ(t) + hb * 16384, &tm_q, &bars[B_Q_FULL], hb * 64, qy + t * kTileRows);
        }
        auto meta = [&](int j, int32_t& ph, int32_t& pp) {
            ph = -1;
            pp = 0;
            if (j < n_ct && lane < kPagesPerTile) {
                const int lp = (t0 + j) * kPagesPerTile + lane;
                if (lp < n_pages) { ph = blk[lp]; pp = page_pos[lp]; }
            }
        };
        int32_t ph_next, pp_next;
        meta(jb, ph_next, pp_next);
        int last[kKStages] = {-1, -1};
        for (int jj = 0; jj < n_loc; ++jj) {
            const int j = jb + jj, ks = jj & 1;
            int32_t ph = ph_next, pp = pp_next;
            meta(j + 1, ph_next, pp_next);
            const bool ok = jj < kKStages || mbar_wait(&bars[B_K_EMPTY + ks], ((jj >> 1) - 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint64_t* full = &bars[B_K_FULL + ks];
            if (j < n_ct) {
                const int np = min(kPagesPerTile, n_pages - (t0 + j) * kPagesPerTile);
                constexpr uint32_t per_page = H * 2048 + (D / 2) * 8;
                if (lane == 0) mbar_arrive_expect_tx(full, per_page * np);
                __syncwarp();
                if (lane < np) {
                    if (ph < 0 || ph >= n_phys) { set_dev_error(kDevErrBounds); ph = 0; }
                    const int32_t y = (ph * Hkv + kvh) * kPage;
#pragma unroll
                    for (int hb = 0; hb < H; ++hb)
                        tma_load_2d(sKs(ks) + hb * 16384 + lane * 2048, &tm_kpool, full, hb * 64, y);
                    bulk_load(sCs(ks) + lane * (D / 2), prm.rope + (int64_t)pp * (D / 2), (D / 2) * 8, full);
                }
            } else if (!LSE && lane == 0) {
                const int32_t fr = row_base + (j - n_ct) * kTileKeys;
                mbar_arrive_expect_tx(full, H * 16384);
                for (int hb = 0; hb < H; ++hb)
                    tma_load_2d(sKs(ks) + hb * 16384, &tm_kfresh, full, hb * 64, kvh * L[L_TOTAL_ROWS] + fr);
            }
            last[ks] = jj;
        }
        if (lane == 0) {
            mbar_drain(&bars[B_Q_FULL], 0);
            for (int s2 = 0; s2 < kKStages; ++s2)
                if (last[s2] >= 0) mbar_drain(&bars[B_K_FULL + s2], (last[s2] >> 1) & 1);
        }
    } else if (warp == kWarpTmaV) {
        // ------------------------------------------------------------ V producer
        if (!LSE) {
            if (lane == 0) {
                prefetch_tmap(&tm_vpool);
                prefetch_tmap(&tm_vfresh);
            }
            auto meta = [&](int j) -> int32_t {
                if (j < n_ct && lane < kPagesPerTile) {
                    const int lp = (t0 + j) * kPagesPerTile + lane;
                    if (lp < n_pages) return blk[lp];
                }
                return -1;
            };
            int32_t ph_next = meta(jb);
            int last[kVStages] = {-1, -1};
            for (int jj = 0; jj < n_loc; ++jj) {
                const int j = jb + jj, vs = jj & 1;
                int32_t ph = ph_next;
                ph_next = meta(j + 1);
                const bool ok = jj < kVStages || mbar_wait(&bars[B_V_EMPTY + vs], ((jj >> 1) - 1) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) break;
                uint64_t* full = &bars[B_V_FULL + vs];
                if (j < n_ct) {
                    const int np = min(kPagesPerTile, n_pages - (t0 + j) * kPagesPerTile);
                    if (lane == 0) mbar_arrive_expect_tx(full, H * 2048 * np);
                    __syncwarp();
                    if (lane < np) {
                        if (ph < 0 || ph >= n_phys) { set_dev_error(kDevErrBounds); ph = 0; }
                        const int32_t y = (ph * Hkv + kvh) * kPage;
#pragma unroll
                        for (int hb = 0; hb < H; ++hb)
                            tma_load_2d(sVs(vs) + hb * 16384 + lane * 2048, &tm_vpool, full, hb * 64, y);
                    }
                } else if (lane == 0) {
                    const int32_t fr = row_base + (j - n_ct) * kTileKeys;
                    mbar_arrive_expect_tx(full, H * 16384);
                    for (int hb = 0; hb < H; ++hb)
                        tma_load_3d(sVs(vs) + hb * 16384, &tm_vfresh, full, hb * 64, kvh, fr);
                }
                last[vs] = jj;
            }
            if (lane == 0)
                for (int s2 = 0; s2 < kVStages; ++s2)
                    if (last[s2] >= 0) mbar_drain(&bars[B_V_FULL + s2], (last[s2] >> 1) & 1);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(128, 128);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 64, true);
            auto issue_qk = [&](int t, int j) {
                const uint32_t aQ = smem_u32(sQ(t)), aK = smem_u32(sKs(j & 1));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = desc_sw128_kmajor(aQ + (kk >> 2) * 16384 + (kk & 3) * 32);
                    const uint64_t b = desc_sw128_kmajor(aK + (kk >> 2) * 16384 + (kk & 3) * 32);
                    mma_bf16_ss(tmem + t * 128, a, b, idesc_qk, kk > 0 ? 1u : 0u);
                }
                // + 1 * bias(key): 0 for taking part, -30000 for excluded / missing keys
                mma_bf16_ss(tmem + t * 128, desc_noswz_kmajor(smem_u32(sQaug), 128, 256),
                            desc_noswz_kmajor(smem_u32(sKaug(j & 1)), 128, 256), idesc_qk, 1u);
                mma_commit(&bars[B_S_FULL + t]);
            };
            auto issue_pv = [&](int t, int j) {
                const uint32_t aV = smem_u32(sVs(j & 1));
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk) {
#pragma unroll
                    for (int nh = 0; nh < H; ++nh) {
                        const uint64_t b = desc_sw128_mn64(aV + nh * 16384 + kk * 2048);
                        mma_bf16_ts(tmem + kTmemO + t * 128 + nh * 64, tmem + t * 128 + kk * 8, b, idesc_pv,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&bars[B_PV_DONE + t]);
            };
            bool ok = mbar_wait(&bars[B_Q_FULL], 0, abort_flag);
            ok = ok && (n_loc == 0 || mbar_wait(&bars[B_KROT_FULL + 0], 0, abort_flag));
            if (ok && n_loc > 0) {
                tc_fence_after();
                issue_qk(0, 0);
                issue_qk(1, 0);
                mma_commit(&bars[B_K_EMPTY + 0]);
            }
            for (int j = 0; ok && j < n_loc; ++j) {    // j: local tile index
                const bool more = j + 1 < n_loc;
                const int kn = (j + 1) & 1;
                if (LSE) {
                    if (more) {
                        ok = mbar_wait(&bars[B_KROT_FULL + kn], ((j + 1) >> 1) & 1, abort_flag);
                        for (int t = 0; ok && t < kQTilesPerCta; ++t) {
                            ok = mbar_wait(&bars[B_S_FREE + t], j & 1, abort_flag);
                            if (!ok) break;
                            tc_fence_after();
                            issue_qk(t, j + 1);
                        }
                        if (ok) mma_commit(&bars[B_K_EMPTY + kn]);
                    }
                    continue;
                }
                // tile A: P_A(j) V(j), then Q_A K(j+1); tile B likewise
                ok = mbar_wait(&bars[B_P_FULL + 0], j & 1, abort_flag) &&
                     mbar_wait(&bars[B_V_FULL + (j & 1)], (j >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(0, j);
                if (more) {
                    ok = mbar_wait(&bars[B_KROT_FULL + kn], ((j + 1) >> 1) & 1, abort_flag) &&
                         mbar_wait(&bars[B_PV_DONE + 0], j & 1, abort_flag);   // P_A columns reused by S_A
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(0, j + 1);
                }
                ok = mbar_wait(&bars[B_P_FULL + 1], j & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(1, j);
                mma_commit(&bars[B_V_EMPTY + (j & 1)]);
                if (more) {
                    ok = mbar_wait(&bars[B_PV_DONE + 1], j & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(1, j + 1);
                    mma_commit(&bars[B_K_EMPTY + kn]);
                }
            }
            mma_commit(&bars[B_DRAIN]);
            mbar_drain(&bars[B_DRAIN], 0);
        }
    } else if (warp >= kWarpRot0) {
        // ------------------------------------------------------------ K rotation (warps 8-11)
        const int rt = tid - kWarpRot0 * 32;
        constexpr int CPR = D / 16;
        constexpr int RGN = kTileKeys / (CPR * kPagesPerTile);
        constexpr int RPT = kPage / RGN;
        const int c = rt % CPR;
        const int rg = rt / (CPR * kPagesPerTile);
        // angle of this thread's first in-page offset (table row rg*RPT) and of one position step
        const float2* cs_start = prm.rope + (rg * RPT) * (D / 2) + 8 * c;
        float2 cs_step[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cs_step[i] = prm.rope[1 * (D / 2) + 8 * c + i];
        // metadata of key rt of the next tile, fetched one tile ahead: logical position and
        // whether the key takes part (cached: page present and token not recomputed; fresh: row
        // present)
        auto meta = [&](int j, int32_t& pos, bool& valid) {
            pos = kNoPos;
            valid = false;
            if (j < n_ct) {
                const int lp = (t0 + j) * kPagesPerTile + rt / kPage;
                if (lp < n_pages) {
                    pos = page_pos[lp] + (rt % kPage);
                    const uint32_t ex = LSE ? 0u : (uint32_t)prm.excl[page_base + lp];
                    valid = ((ex >> (rt % kPage)) & 1u) == 0u;
                }
            } else if (j < n_tiles) {
                const int fr = (j - n_ct) * kTileKeys + rt;
                if (fr < n_rows_req) { pos = prm.row_pos[row_base + fr]; valid = true; }
            }
        };
        int32_t pos_n;
        bool val_n;
        meta(jb, pos_n, val_n);
        for (int jj = 0; jj < n_loc; ++jj) {
            const int j = jb + jj, ks = jj & 1;
            const int32_t pos = pos_n;
            const bool val = val_n;
            meta(j + 1, pos_n, val_n);
            bool ok = mbar_wait(&bars[B_K_FULL + ks], (jj >> 1) & 1, abort_flag);
            ok = ok && (jj < kKStages || mbar_wait(&bars[B_KPOS_FREE + ks], ((jj >> 1) - 1) & 1, abort_flag));
            if (!__all_sync(0xffffffffu, ok)) break;
            if (j < n_ct) rotate_cached_tile<D>(sKs(ks), sCs(ks), rt, cs_start, cs_step);
            sKpos(ks)[rt] = pos;
            *reinterpret_cast<__half*>(sKaug(ks) + slab16_off(rt, 0)) = __float2half(val ? 0.f : kKeyOff);
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_KROT_FULL + ks]);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-7)
        // Group t (warps 4t..4t+3) owns Q tile t.  Scores arrive already in log2 units: the
        // rotated query rows carry log2(e)/sqrt(d).
        const int t = warp >= kWarpSoftB ? 1 : 0;
        const int m = tid - t * 128;           // tile row = TMEM lane
        const int tok = m / g, hl = m % g;
        const int row = row0 + t * toks_per_tile + tok;
        const bool valid = row < n_rows_req;
        int32_t mypos;
        if (LSE) mypos = valid ? kNoPos - 1 : -1;
        else mypos = valid ? prm.row_pos[row_base + row] : -1;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_addr + t * 128;          // S (and P) columns of this tile
        const uint32_t tO = tmem + lane_addr + kTmemO + t * 128;
        // output locations, fixed before the tile loop so that only one pointer stays live across it
        // (a split key range writes a normalized partial row plus its max and sum instead)
        __nv_bfloat16* out_row = nullptr;
        float2* ml_slot = nullptr;
        if (valid) {
            if (LSE) {
                ml_slot = prm.lse_part + R[R_LSE_BASE] +
                          ((int64_t)kvh * (R[R_N_QUERY] * g) + row * g + hl) * R[R_LSE_CHUNKS] + chunk;
            } else if (R[R_NSPLIT] == 1) {
                out_row = prm.out + ((int64_t)(row_base + row) * Hq + kvh * g + hl) * D;
            } else {
                const int64_t prow = (int64_t)(R[R_SLOT_BASE] + (kvh * R[R_NPAIRS] + qpair) * R[R_NSPLIT] + chunk) *
                                         (kQTilesPerCta * kTileRows) + t * kTileRows + m;
                out_row = prm.part_o + prow * D;
                ml_slot = prm.part_ml + prow;
            }
        }
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_loc; ++j) {    // j: local tile index
            const int ks = j & 1;
            ok = mbar_wait(&bars[B_S_FULL + t], j & 1, abort_flag);
            ok = ok && mbar_wait(&bars[B_KROT_FULL + ks], (j >> 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // causal limit of this row inside the tile: keys are in increasing position order, so
            // the visible ones are a prefix (binary search); excluded keys are already at -30000
            int cut;
            {
                const int32_t* kp = sKpos(ks);
                int lo = 0;
#pragma unroll
                for (int step = 64; step >= 1; step >>= 1)
                    if (kp[lo + step - 1] <= mypos) lo += step;
                if (kp[lo] <= mypos) ++lo;   // lo <= 127 here; 128 when every key qualifies
                cut = lo;
            }
            mbar_arrive(&bars[B_KPOS_FREE + ks]);
            const bool full = __all_sync(0xffffffffu, cut == kTileKeys);   // no row of the warp is cut
            // pass 1: row max
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t sv[32];
                tmem_ld32(tS + cc * 32, sv);
                tmem_ld_wait();
                if (full) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        mx4[0] = max3f(mx4[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                        mx4[1] = max3f(mx4[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                        mx4[2] = max3f(mx4[2], __uint_as_float(sv[e + 4]), __uint_as_float(sv[e + 5]));
                        mx4[3] = max3f(mx4[3], __uint_as_float(sv[e + 6]), __uint_as_float(sv[e + 7]));
                    }
                } else {
                    const int k = cut - 32 * cc;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float x = e < k ? __uint_as_float(sv[e]) : -INFINITY;
                        mx4[e & 3] = fmaxf(mx4[e & 3], x);
                    }
                }
            }
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            const float m_new = fmaxf(m_run, mx);
            const bool need = m_new > m_run + 8.0f;     // lazy rescale: keep P <= 2^8
            const float alpha = need ? ex2(m_run - m_new) : 1.0f;
            if (need) { l_run *= alpha; m_run = m_new; }
            const float msub = m_run == -INFINITY ? 0.f : m_run;
            if (!LSE && j > 0) {
                // PV(j-1) of this tile must be done before O is rescaled
                ok = mbar_wait(&bars[B_PV_DONE + t], (j - 1) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
            }
            // pass 2: p = 2^(s - m) for visible keys; P (bf16 pairs) overwrites the S columns
            // already read (columns [16cc, 16cc+16) after S columns [32cc, 32cc+32) are loaded)
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t sv[32], pk[16];
                tmem_ld32(tS + cc * 32, sv);
                tmem_ld_wait();
                if (full) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = ex2(__uint_as_float(sv[2 * e]) - msub);
                        const float p1 = ex2(__uint_as_float(sv[2 * e + 1]) - msub);
                        sum4[e & 3] += p0 + p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                } else {
                    const int k = cut - 32 * cc;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = 2 * e < k ? ex2(__uint_as_float(sv[2 * e]) - msub) : 0.f;
                        const float p1 = 2 * e + 1 < k ? ex2(__uint_as_float(sv[2 * e + 1]) - msub) : 0.f;
                        sum4[e & 3] += p0 + p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                }
                if (!LSE) tmem_st16(tS + cc * 16, pk);
            }
            l_run += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
            if (LSE) {
                tc_fence_before();
                mbar_arrive(&bars[B_S_FREE + t]);
            } else {
                if (j > 0 && __any_sync(0xffffffffu, need)) {
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
                mbar_arrive(&bars[B_P_FULL + t]);
            }
        }
        if (ml_slot != nullptr && ok) *ml_slot = make_float2(n_loc > 0 ? m_run : -INFINITY, l_run);
        if (!LSE && ok && n_loc > 0) {
            ok = mbar_wait(&bars[B_PV_DONE + t], (n_loc - 1) & 1, abort_flag);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + cc * 32, o);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                            *reinterpret_cast<uint4*>(out_row + cc * 32 + 8 * q) = w;
                        }
                    }
                }
            }
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
