// Flash-style attention over the position-free paged cache with in-kernel RoPE (sm_103a).
//
// MiniPIC, section 2.1: cached keys k~_j stay unrotated in shared pages; the attention kernel
// rotates them on the fly to the key's per-request logical position pi(j) with a cos/sin lookup
// and fused multiply-adds, so score(t, j) = (R_t q_t)^T (R_pi(j) k~_j) / sqrt(d).
// QCFuse, section 2C / Phase 4 (and the sparse attention kernel of its section 3): the recomputed
// tokens and the query tokens attend over the cached keys minus the recomputed ones plus the
// fresh rows, keeping causal order on logical positions.
//
// One CTA = one tile of 128 query rows (the g query heads of 128/g consecutive rows of one
// request, all sharing kv head `kvh`) against the request's KV tiles of 128 keys:
//   warps 0-3  softmax: S row from TMEM, mask, online softmax (lazy rescale), P -> smem, O epilogue
//   warp  4    TMEM allocation + single-thread tcgen05.mma issue
//   warp  5    TMA producer: Q tile, cached K/V pages through the block table, page cos/sin rows,
//              fresh K/V tiles
//   warps 6-9  rotate cached K tiles in shared memory (in place, 128-byte swizzled K-major)
// S = Q K^T (M=128, N=128, K=d) is double-buffered in TMEM; O (M=128, N=d) accumulates in TMEM.
// Cached keys are rotated by composing the page-base angle (cos/sin row of the page's first
// position, copied per page) with the in-page offset, advanced row by row (angle addition).
// LSE mode (critical-layer scoring, pass 1) runs the same pipeline without P/V and writes the
// per-row running max and sum of one key chunk.
#pragma once
#include "layout_format.h"
#include "ptx.cuh"

namespace pcf {

constexpr int kAttnThreads = 320;
constexpr int kWarpMma = 4;
constexpr int kWarpTma = 5;
constexpr int kWarpRot0 = 6;
constexpr int kNoPos = 0x7FFFFFFF;

struct AttnParams {
    const int32_t* layout;
    const uint16_t* excl;      // attention: per logical page exclusion bits
    const int32_t* row_pos;    // attention: logical position of every row
    const float2* rope;        // [max_pos][D/2] (cos, sin)
    __nv_bfloat16* out;        // attention: [rows][Hq][D]
    float2* lse_part;          // LSE: (running max in log2 units, running sum) per row and chunk
    float scale_log2;          // log2(e) / sqrt(D)
};

template <int D, bool LSE>
struct AttnSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kQ = kTileRows * D * 2;
    static constexpr int kK = kTileKeys * D * 2;
    static constexpr int kV = LSE ? 0 : kTileKeys * D * 2;
    static constexpr int kP = LSE ? 0 : kTileRows * kTileKeys * 2;
    static constexpr int kCs = kPagesPerTile * (D / 2) * 8;
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kQ;
    static constexpr int oV = oK + 2 * kK;
    static constexpr int oP = oV + 2 * kV;
    static constexpr int oCs = oP + kP;
    static constexpr int oKpos = oCs + 2 * kCs;
    static constexpr int oBar = oKpos + 2 * kTileKeys * 4;
    static constexpr int kNumBars = 16;
    static constexpr int oMisc = oBar + kNumBars * 8;
    static constexpr int kBytes = oMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;   // slack for 1024-byte alignment
    static constexpr uint32_t kTmemCols = LSE ? 256 : 512;
};

// barrier slots
enum : int {
    B_Q_FULL = 0, B_TMA_FULL = 1 /*2*/, B_KROT_FULL = 3 /*2*/, B_KV_EMPTY = 5 /*2*/, B_S_FULL = 7 /*2*/,
    B_S_FREE = 9 /*2*/, B_KPOS_FREE = 11 /*2*/, B_P_FULL = 13, B_P_FREE = 14, B_DRAIN = 15
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
// c of rows rg*RPT .. rg*RPT+RPT-1 of page pg; it composes the page-base angle with its first
// row's offset once and then advances the angle by one position per row.
// Writes key_pos (INT_MAX for missing or excluded tokens).
template <int D>
__device__ __forceinline__ int rot_page_of(int rt) { return (rt / (D / 16)) % kPagesPerTile; }
// `p0` / `ex`: logical position of the page's first token and its exclusion bits (prefetched by
// the caller one tile ahead); `page_valid` false for pages past the request's end.
template <int D>
__device__ __forceinline__ void rotate_cached_tile(uint8_t* sK, const float2* sCs, int32_t* kpos, int rt,
                                                   bool page_valid, int32_t p0, uint32_t ex,
                                                   const float2 (&cs_start)[8], const float2 (&cs_step)[8]) {
    constexpr int CPR = D / 16;
    constexpr int RGN = kTileKeys / (CPR * kPagesPerTile);
    constexpr int RPT = kPage / RGN;
    const int c = rt % CPR;
    const int pg = (rt / CPR) % kPagesPerTile;
    const int rg = rt / (CPR * kPagesPerTile);
    const int row0 = pg * kPage + rg * RPT;
    if (page_valid) {
        float2 cs[8];
        const float4* b4 = reinterpret_cast<const float4*>(sCs + pg * (D / 2) + 8 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = b4[q];
            cs[2 * q] = cmul(make_float2(v.x, v.y), cs_start[2 * q]);
            cs[2 * q + 1] = cmul(make_float2(v.z, v.w), cs_start[2 * q + 1]);
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int off = rg * RPT + r;
            const bool dropped = (ex >> off) & 1u;
            if (!dropped) rotate_chunk_pair<D>(sK, row0 + r, c, cs);
            if (c == 0) kpos[row0 + r] = dropped ? kNoPos : p0 + off;
#pragma unroll
            for (int i = 0; i < 8; ++i) cs[i] = cmul(cs[i], cs_step[i]);
        }
    } else if (c == 0) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) kpos[row0 + r] = kNoPos;
    }
}

template <int D, bool LSE>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kpool,
            const __grid_constant__ CUtensorMap tm_vpool, const __grid_constant__ CUtensorMap tm_kfresh,
            const __grid_constant__ CUtensorMap tm_vfresh, const AttnParams prm) {
    using SM = AttnSmem<D, LSE>;
    constexpr int H = SM::kHalves;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + SM::oQ;
    auto sKs = [&](int st) { return smem + SM::oK + st * SM::kK; };
    auto sVs = [&](int st) { return smem + SM::oV + st * SM::kV; };
    uint8_t* sP = smem + SM::oP;
    auto sCs = [&](int st) { return reinterpret_cast<float2*>(smem + SM::oCs + st * SM::kCs); };
    auto sKpos = [&](int st) { return reinterpret_cast<int32_t*>(smem + SM::oKpos) + st * kTileKeys; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::oBar);
    int32_t* misc = reinterpret_cast<int32_t*>(smem + SM::oMisc);
    // misc: [0] tmem base, [1] n cached tiles, [2] n fresh tiles, [3] first cached tile, [4] abort
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* L = prm.layout;
    const int32_t* item = L + (LSE ? L[L_OFF_LSE] : L[L_OFF_ATTN]) + kItemWords * blockIdx.x;
    const int req = item[0], kvh = item[1], qt = item[2], chunk = item[3];
    const int32_t* R = L + L[L_OFF_REQ] + req * R_STRIDE;
    const int Hq = L[L_HQ], Hkv = L[L_HKV], g = L[L_GROUP];
    const int toks_per_tile = kTileRows / g;
    const int n_rows_req = LSE ? R[R_N_QUERY] : R[R_N_ROWS];
    const int row0 = qt * toks_per_tile;
    const int ntok = min(toks_per_tile, n_rows_req - row0);
    const int n_pages = R[R_N_PAGES];
    const int32_t page_base = R[R_PAGE_BASE];
    const int32_t row_base = R[R_ROW_BASE];
    const int32_t* page_pos = L + L[L_OFF_PAGEPOS] + page_base;
    const int32_t* blk = L + L[L_OFF_BLOCK] + page_base;

    if (tid == 0) {
        mbar_init(&bars[B_Q_FULL], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_TMA_FULL + s], 1);
            mbar_init(&bars[B_KROT_FULL + s], 128);
            mbar_init(&bars[B_KV_EMPTY + s], 1);
            mbar_init(&bars[B_S_FULL + s], 1);
            mbar_init(&bars[B_S_FREE + s], 128);
            mbar_init(&bars[B_KPOS_FREE + s], 128);
        }
        mbar_init(&bars[B_P_FULL], 128);
        mbar_init(&bars[B_P_FREE], 1);
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
            const int32_t pmax = ntok > 0 ? prm.row_pos[row_base + row0 + ntok - 1] : -1;
            nct = 0;
            while (nct < nkt && page_pos[nct * kPagesPerTile] <= pmax) ++nct;
            const int nft_total = (n_rows_req + kTileKeys - 1) / kTileKeys;
            while (nft < nft_total && prm.row_pos[row_base + nft * kTileKeys] <= pmax) ++nft;
        }
        misc[1] = nct;
        misc[2] = nft;
        misc[3] = t0;
        misc[4] = 0;
    }
    if (warp == kWarpMma) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), SM::kTmemCols);
        tmem_relinquish();
    }
    // V stages and the P buffer start finite: masked keys contribute 0 * V
    if (!LSE) {
        uint4* z = reinterpret_cast<uint4*>(smem + SM::oV);
        for (int i = tid; i < (2 * SM::kV) / 16; i += kAttnThreads) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);
    const int n_ct = misc[1], n_ft = misc[2], t0 = misc[3];
    const int n_tiles = n_ct + n_ft;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer
        // Lane p (< 8) fetches the block-table entry and position of page p of the next tile while
        // the current one is issued, then issues that page's copies itself.
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_kpool);
            if (!LSE) {
                prefetch_tmap(&tm_vpool);
                prefetch_tmap(&tm_kfresh);
                prefetch_tmap(&tm_vfresh);
            }
            const int32_t qy = LSE ? (kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE] + row0) * g
                                   : (kvh * L[L_TOTAL_ROWS] + row_base + row0) * g;
            mbar_arrive_expect_tx(&bars[B_Q_FULL], SM::kQ);
            for (int hb = 0; hb < H; ++hb) tma_load_2d(sQ + hb * 16384, &tm_q, &bars[B_Q_FULL], hb * 64, qy);
        }
        const int n_phys = L[L_N_PHYS];
        auto meta = [&](int j, int32_t& ph, int32_t& pp) {
            ph = -1;
            pp = 0;
            if (j < n_ct && lane < kPagesPerTile) {
                const int lp = (t0 + j) * kPagesPerTile + lane;
                if (lp < n_pages) { ph = blk[lp]; pp = page_pos[lp]; }
            }
        };
        int32_t ph_next, pp_next;
        meta(0, ph_next, pp_next);
        int last[2] = {-1, -1};
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            int32_t ph = ph_next, pp = pp_next;
            meta(j + 1, ph_next, pp_next);
            bool ok = j < 2 || mbar_wait(&bars[B_KV_EMPTY + st], ((j >> 1) - 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint64_t* full = &bars[B_TMA_FULL + st];
            if (j < n_ct) {
                const int np = min(kPagesPerTile, n_pages - (t0 + j) * kPagesPerTile);
                constexpr uint32_t per_page = H * 2048 * (LSE ? 1 : 2) + (D / 2) * 8;
                if (lane == 0) mbar_arrive_expect_tx(full, per_page * np);
                __syncwarp();
                if (lane < np) {
                    if (ph < 0 || ph >= n_phys) { set_dev_error(kDevErrBounds); ph = 0; }
                    const int32_t y = (ph * Hkv + kvh) * kPage;
#pragma unroll
                    for (int hb = 0; hb < H; ++hb) {
                        tma_load_2d(sKs(st) + hb * 16384 + lane * 2048, &tm_kpool, full, hb * 64, y);
                        if (!LSE) tma_load_2d(sVs(st) + hb * 16384 + lane * 2048, &tm_vpool, full, hb * 64, y);
                    }
                    bulk_load(sCs(st) + lane * (D / 2), prm.rope + (int64_t)pp * (D / 2), (D / 2) * 8, full);
                }
            } else if (!LSE && lane == 0) {
                const int32_t fr = row_base + (j - n_ct) * kTileKeys;
                mbar_arrive_expect_tx(full, H * 16384 * 2);
                for (int hb = 0; hb < H; ++hb) {
                    tma_load_2d(sKs(st) + hb * 16384, &tm_kfresh, full, hb * 64, kvh * L[L_TOTAL_ROWS] + fr);
                    tma_load_3d(sVs(st) + hb * 16384, &tm_vfresh, full, hb * 64, kvh, fr);
                }
            }
            last[st] = j;
        }
        if (lane == 0) {
            mbar_drain(&bars[B_Q_FULL], 0);
            for (int s2 = 0; s2 < 2; ++s2)
                if (last[s2] >= 0) mbar_drain(&bars[B_TMA_FULL + s2], (last[s2] >> 1) & 1);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(128, 128);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 64, true);
            const uint32_t aQ = smem_u32(sQ);
            const uint32_t aP = smem_u32(sP);
            bool ok = mbar_wait(&bars[B_Q_FULL], 0, abort_flag);
            auto issue_pv = [&](int i) -> bool {
                if (!mbar_wait(&bars[B_P_FULL], i & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t aV = smem_u32(sVs(i & 1));
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                    const uint64_t a = desc_sw128_kmajor(aP + (kk >> 2) * 16384 + (kk & 3) * 32);
#pragma unroll
                    for (int nh = 0; nh < H; ++nh) {
                        const uint64_t b = desc_sw128_mn64(aV + nh * 16384 + kk * 2048);
                        mma_bf16_ss(tmem + 256 + nh * 64, a, b, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&bars[B_P_FREE]);
                mma_commit(&bars[B_KV_EMPTY + (i & 1)]);
                return true;
            };
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int st = j & 1;
                if (!mbar_wait(&bars[B_KROT_FULL + st], (j >> 1) & 1, abort_flag)) { ok = false; break; }
                if (j >= 2 && !mbar_wait(&bars[B_S_FREE + st], ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t aK = smem_u32(sKs(st));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = desc_sw128_kmajor(aQ + (kk >> 2) * 16384 + (kk & 3) * 32);
                    const uint64_t b = desc_sw128_kmajor(aK + (kk >> 2) * 16384 + (kk & 3) * 32);
                    mma_bf16_ss(tmem + st * 128, a, b, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars[B_S_FULL + st]);
                if (LSE) mma_commit(&bars[B_KV_EMPTY + st]);
                else if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (!LSE && ok && n_tiles > 0) issue_pv(n_tiles - 1);
            mma_commit(&bars[B_DRAIN]);
            mbar_drain(&bars[B_DRAIN], 0);
        }
    } else if (warp >= kWarpRot0) {
        // ------------------------------------------------------------ K rotation
        const int rt = tid - kWarpRot0 * 32;
        constexpr int CPR = D / 16;
        constexpr int RGN = kTileKeys / (CPR * kPagesPerTile);
        constexpr int RPT = kPage / RGN;
        const int c = rt % CPR;
        const int rg = rt / (CPR * kPagesPerTile);
        float2 cs_start[8], cs_step[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            cs_start[i] = prm.rope[(rg * RPT) * (D / 2) + 8 * c + i];
            cs_step[i] = prm.rope[1 * (D / 2) + 8 * c + i];
        }
        const int pg = rot_page_of<D>(rt);
        // metadata of the next tile, fetched one tile ahead: cached tiles (page position, exclusion
        // bits of this thread's page), fresh tiles (position of key rt)
        auto meta = [&](int j, int32_t& m0, uint32_t& m1) {
            m0 = kNoPos;
            m1 = 0u;
            if (j < n_ct) {
                const int lp = (t0 + j) * kPagesPerTile + pg;
                if (lp < n_pages) {
                    m0 = page_pos[lp];
                    m1 = LSE ? 0u : (uint32_t)prm.excl[page_base + lp];
                }
            } else if (j < n_tiles) {
                const int fr = (j - n_ct) * kTileKeys + rt;
                if (fr < n_rows_req) m0 = prm.row_pos[row_base + fr];
            }
        };
        int32_t m0n;
        uint32_t m1n;
        meta(0, m0n, m1n);
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            const int32_t m0 = m0n;
            const uint32_t m1 = m1n;
            meta(j + 1, m0n, m1n);
            if (!mbar_wait(&bars[B_TMA_FULL + st], (j >> 1) & 1, abort_flag)) break;
            if (j >= 2 && !mbar_wait(&bars[B_KPOS_FREE + st], ((j >> 1) - 1) & 1, abort_flag)) break;
            if (j < n_ct) {
                const bool pv = (t0 + j) * kPagesPerTile + pg < n_pages;
                rotate_cached_tile<D>(sKs(st), sCs(st), sKpos(st), rt, pv, m0, m1, cs_start, cs_step);
            } else {
                sKpos(st)[rt] = m0;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_KROT_FULL + st]);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-3)
        const int m = tid;                 // tile row = TMEM lane
        const int tok = m / g, hl = m % g;
        const bool valid = tok < ntok;
        const int row = row0 + tok;
        int32_t mypos;
        if (LSE) mypos = valid ? kNoPos - 1 : -1;
        else mypos = valid ? prm.row_pos[row_base + row] : -1;
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const float scale = prm.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            ok = mbar_wait(&bars[B_S_FULL + st], (j >> 1) & 1, abort_flag);
            ok = ok && mbar_wait(&bars[B_KROT_FULL + st], (j >> 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t sv[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_addr + st * 128 + cc * 32, sv[cc]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bars[B_S_FREE + st]);
            float mx = -INFINITY;
            const int4* kp4 = reinterpret_cast<const int4*>(sKpos(st));
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int4 kp = kp4[q];
                const int cc = q >> 3, e = (q & 7) * 4;
                float v0 = kp.x <= mypos ? __uint_as_float(sv[cc][e + 0]) * scale : -INFINITY;
                float v1 = kp.y <= mypos ? __uint_as_float(sv[cc][e + 1]) * scale : -INFINITY;
                float v2 = kp.z <= mypos ? __uint_as_float(sv[cc][e + 2]) * scale : -INFINITY;
                float v3 = kp.w <= mypos ? __uint_as_float(sv[cc][e + 3]) * scale : -INFINITY;
                mx = fmaxf(mx, fmaxf(fmaxf(v0, v1), fmaxf(v2, v3)));
                sv[cc][e + 0] = __float_as_uint(v0);
                sv[cc][e + 1] = __float_as_uint(v1);
                sv[cc][e + 2] = __float_as_uint(v2);
                sv[cc][e + 3] = __float_as_uint(v3);
            }
            mbar_arrive(&bars[B_KPOS_FREE + st]);
            const float m_new = fmaxf(m_run, mx);
            const bool need = m_new > m_run + 8.0f;     // lazy rescale: keep P <= 2^8
            const float alpha = need ? ex2(m_run - m_new) : 1.0f;
            if (need) { l_run *= alpha; m_run = m_new; }
            const float msub = m_run == -INFINITY ? 0.f : m_run;
            if (!LSE && j > 0) {
                // PV_{j-1} must be done: it reads the single P buffer and accumulates into O
                ok = mbar_wait(&bars[B_P_FREE], (j - 1) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
            }
            float sum = 0.f;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const int cc = ch >> 2, e = (ch & 3) * 8;
                float p[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    p[u] = ex2(__uint_as_float(sv[cc][e + u]) - msub);
                    sum += p[u];
                }
                if (!LSE) {
                    uint4 w;
                    w.x = pack_bf16x2(p[0], p[1]);
                    w.y = pack_bf16x2(p[2], p[3]);
                    w.z = pack_bf16x2(p[4], p[5]);
                    w.w = pack_bf16x2(p[6], p[7]);
                    *reinterpret_cast<uint4*>(sP + (ch >> 3) * 16384 + sw128_off(m, ch & 7)) = w;
                }
            }
            l_run += sum;
            if (!LSE) {
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_addr + 256 + cc * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_addr + 256 + cc * 32, o);
                    }
                    tmem_st_wait();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars[B_P_FULL]);
            }
        }
        if (LSE) {
            if (ok && valid) {
                const int chunks = R[R_LSE_CHUNKS];
                const int n_q = R[R_N_QUERY] * g;
                prm.lse_part[R[R_LSE_BASE] + ((int64_t)kvh * n_q + row * g + hl) * chunks + chunk] =
                    make_float2(m_run, l_run);
            }
        } else if (ok && n_tiles > 0) {
            ok = mbar_wait(&bars[B_P_FREE], (n_tiles - 1) & 1, abort_flag);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
                __nv_bfloat16* dst = prm.out + ((int64_t)(row_base + row) * Hq + kvh * g + hl) * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_addr + 256 + cc * 32, o);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                            *reinterpret_cast<uint4*>(dst + cc * 32 + 8 * q) = w;
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
