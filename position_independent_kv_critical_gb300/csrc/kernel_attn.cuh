// Flash-style attention over the position-free paged cache (sm_103a).
//
// MiniPIC, section 2.1: cached keys k~_j stay unrotated in shared pages and are rotated at use time
// to the key's per-request logical position pi(j), so score(t, j) = (R_t q_t)^T (R_pi(j) k~_j) /
// sqrt(d).  The rotation of a request's cached keys runs once per call (rope_rows_kernel in page
// gather mode, into the call's workspace) rather than inside this kernel: a cached key tile is
// visited by every 256-row query block of the request, and rotating it there costs more than
// writing and re-reading the rotated tile once.
// QCFuse, section 2C / Phase 4 (and the sparse attention kernel of its section 3): the recomputed
// tokens and the query tokens attend over the cached keys minus the recomputed ones plus the
// fresh rows, keeping causal order on logical positions.
//
// One CTA = two tiles A and B of 128 query rows each (a tile packs the g query heads of 128/g
// consecutive rows of one request, all sharing kv head `kvh`) against the request's KV tiles of
// 128 keys; both tiles share every K and V tile:
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: S row from TMEM, causal cut,
//               online softmax (lazy rescale), P -> TMEM (over the S columns), O epilogue
//   warps 8/11  Q K^T issue for tile A / B (warp 8 also owns the TMEM allocation)
//   warps 12/13 P V issue for tile A / B.  Each key tile is processed in two 64-key halves
//               q = 2j, 2j+1 and S is double-buffered per query tile: P(q) V runs, then Q K(q+2)
//               goes into the buffer P(q) came from, while the softmax already works on S(q+1).
//               Four single-thread issuers keep four independent MMA streams in flight: one
//               thread's stream of 128-row MMAs with N <= 128 is bound by per-instruction
//               latency, not by the tensor core's rate
//   warp  9     K producer: rotated K tiles (compacted cached or fresh, fp16, TMA) and, per
//               key, its logical position; 2-stage ring, freed by the second half's Q K^T
//   (warp 0 starts the Q tile loads during set-up)
//   warp  10    V producer (TMA): compacted cached V tiles / fresh V tiles; 2-stage ring, freed
//               once both P V of a stage are done
// TMEM: tile t's two S half-buffers at columns t*128 + {0, 64} (64 fp32 columns = 64 keys each),
// O_A at [256,256+d), O_B at [384,384+d).  S = Q K^T is fp16 x fp16 (M=128, N=64 keys, K=d); P
// (bf16 pairs, 32 columns) overwrites the S half it came from and is the A operand of
// O += P V (M=128, N=d in one instruction, K=64 keys, V as an MN-major bf16 operand whose two
// 64-wide halves are 16 KB apart).
// The cached keys arrive compacted: recomputed tokens' cached copies are left out of the rotated
// K/V copy, so every cached key streamed takes part.  Key positions increase along the cached
// keys and along the fresh rows, and missing keys (past a ragged end) carry position kNoPos, so a
// row's visible keys in a tile are a prefix of it; only rows whose causal limit falls inside a
// tile need per-element masking.
// LSE mode (critical-layer scoring, pass 1) runs the same pipeline without P/V and writes the
// per-row running max and sum of one key chunk.
#pragma once
#include "layout_format.h"
#include "ptx.cuh"

namespace pcf {

constexpr int kAttnThreads = 448;   // 14 warps: at most 4 per SM sub-partition (128 registers)
constexpr int kWarpSoftB = 4;
constexpr int kWarpMma = 8;
constexpr int kWarpTma = 9;
constexpr int kWarpTmaV = 10;
constexpr int kWarpMmaB = 11;
constexpr int kWarpPvA = 12;
constexpr int kWarpPvB = 13;
constexpr int kNoPos = 0x7FFFFFFF;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kTmemO = 256;     // O_A at 256, O_B at 384

struct AttnParams {
    const int32_t* layout;
    const int32_t* kpos_c;     // attention: logical position of every compacted cached key
    const int32_t* row_pos;    // attention: logical position of every row
    __nv_bfloat16* out;        // attention: [rows][Hq][D]
    float2* lse_part;          // LSE: (running max in log2 units, running sum) per row and chunk
    float* lse_final;          // LSE: log2-sum-exp per row, [Hkv][total query][g]
    int32_t* lse_count;        // LSE: finished chunks per (request, kv head, pair); zero on entry and exit
    __nv_bfloat16* part_o;     // attention with a split key range: normalized partial O per slot
    float2* part_ml;           //   and its (running max, running sum) per row
};

template <int D, bool LSE>
struct AttnSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kQ = kTileRows * D * 2;          // one Q tile
    static constexpr int kK = kTileKeys * D * 2;
    static constexpr int kV = LSE ? 0 : kTileKeys * D * 2;
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kQTilesPerCta * kQ;
    static constexpr int oV = oK + kKStages * kK;
    static constexpr int oKpos = oV + kVStages * kV;
    static constexpr int oBar = oKpos + kKStages * kTileKeys * 4;
    static constexpr int kNumBars = 30;
    static constexpr int oMisc = oBar + kNumBars * 8;
    static constexpr int kBytes = oMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;   // slack for 1024-byte alignment
    static constexpr uint32_t kTmemCols = LSE ? 256 : 512;
};

// barrier slots
enum : int {
    B_Q_FULL = 0,
    B_K_FULL = 1,      // [2] rotated K tile landed and its key positions / biases written
    B_K_EMPTY = 3,     // [2] both Q K^T that read the stage are done (one commit per issuer)
    B_KPOS_FREE = 5,   // [2] both softmax groups are done with the stage's key info (256 arrivals)
    B_V_FULL = 7,      // [2]
    B_V_EMPTY = 9,     // [2] both P V that read the stage are done (one commit per issuer)
    B_S_FULL = 11,     // [4] per (Q tile, S half-buffer): S = Q K^T of a 64-key half landed
    B_P_FULL = 15,     // [4] per (Q tile, S half-buffer): P written and O rescaled; in LSE mode:
                       //     softmax done reading that S half
    B_PV_DONE = 19,    // [4] per (Q tile, S half-buffer): P V of that buffer's latest half is done
    B_O_DONE = 23,     // [2] per Q tile: the last P V is done (single phase)
    B_DRAIN = 25       // [4] per issuer: its last MMA is done
};

template <int D, bool LSE>
__global__ void __launch_bounds__(kAttnThreads)
attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kcache,
            const __grid_constant__ CUtensorMap tm_vcache, const __grid_constant__ CUtensorMap tm_kfresh,
            const __grid_constant__ CUtensorMap tm_vfresh, const AttnParams prm) {
    using SM = AttnSmem<D, LSE>;
    constexpr int H = SM::kHalves;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sQ = [&](int t) { return smem + SM::oQ + t * SM::kQ; };
    auto sKs = [&](int st) { return smem + SM::oK + st * SM::kK; };
    auto sVs = [&](int st) { return smem + SM::oV + st * SM::kV; };
    auto sKpos = [&](int st) { return reinterpret_cast<int32_t*>(smem + SM::oKpos) + st * kTileKeys; };
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
    const int32_t* PR = L + L[L_OFF_PAIR] + (R[R_PAIR_BASE] + qpair) * P_STRIDE;   // attention only
    const int Hq = L[L_HQ], Hkv = L[L_HKV], g = L[L_GROUP];
    const int toks_per_tile = kTileRows / g;
    const int n_rows_req = LSE ? R[R_N_QUERY] : R[R_N_ROWS];
    const int row0 = qpair * kQTilesPerCta * toks_per_tile;        // first row of tile A
    const int nrow_cta = min(kQTilesPerCta * toks_per_tile, n_rows_req - row0);
    const int n_pages = R[R_N_PAGES];
    const int32_t page_base = R[R_PAGE_BASE];
    const int32_t row_base = R[R_ROW_BASE];
    const int32_t* page_pos = L + L[L_OFF_PAGEPOS] + page_base;

    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&bars[B_Q_FULL], 1);
            for (int s2 = 0; s2 < kKStages; ++s2) {
                mbar_init(&bars[B_K_FULL + s2], 32);   // every producer lane (key info) + TMA bytes
                mbar_init(&bars[B_K_EMPTY + s2], kQTilesPerCta);
                mbar_init(&bars[B_KPOS_FREE + s2], 256);
            }
            for (int s2 = 0; s2 < kVStages; ++s2) {
                mbar_init(&bars[B_V_FULL + s2], 1);
                mbar_init(&bars[B_V_EMPTY + s2], kQTilesPerCta);
            }
            for (int t = 0; t < kQTilesPerCta; ++t) {
                for (int b = 0; b < 2; ++b) {
                    mbar_init(&bars[B_S_FULL + 2 * t + b], 1);
                    mbar_init(&bars[B_P_FULL + 2 * t + b], 128);
                }
                mbar_init(&bars[B_PV_DONE + 2 * t], 1);
                mbar_init(&bars[B_PV_DONE + 2 * t + 1], 1);
                mbar_init(&bars[B_O_DONE + t], 1);
            }
            for (int i = 0; i < 2 * kQTilesPerCta; ++i) mbar_init(&bars[B_DRAIN + i], 1);
            fence_mbar_init();
            prefetch_tmap(&tm_q);
        }
    }
    // up to here only the layout and shared memory were touched: the previous kernel (which
    // writes the rotated rows, the compacted keys and their positions) may still be running
    grid_dep_wait();
    grid_dep_launch();
    if (warp == 0) {
        if (lane == 0) {
            // the Q tiles do not depend on the key range: start them before it is computed
            const int32_t qy = LSE ? (kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE] + row0) * g
                                   : (kvh * L[L_TOTAL_ROWS] + row_base + row0) * g;
            mbar_arrive_expect_tx(&bars[B_Q_FULL], kQTilesPerCta * SM::kQ);
            for (int t = 0; t < kQTilesPerCta; ++t)
                for (int hb = 0; hb < H; ++hb)
                    tma_load_2d(sQ(t) + hb * 16384, &tm_q, &bars[B_Q_FULL], hb * 64, qy + t * kTileRows);
        }
        int nct = 0, nft = 0, t0 = 0;
        // LSE: tiles of all the request's cached tokens; attention: tiles of the compacted ones
        const int nkt = LSE ? R[R_N_KTILES] : (n_pages * kPage - R[R_N_SEL] + kTileKeys - 1) / kTileKeys;
        if (LSE) {
            const int chunks = R[R_LSE_CHUNKS];
            const int tpc = (nkt + chunks - 1) / chunks;
            t0 = chunk * tpc;
            nct = max(0, min(tpc, nkt - t0));
        } else {
            // visible tiles: key positions increase along the cached tiles and along the fresh rows,
            // so each count is the number of tiles whose first key is at or before the CTA's last
            // row (the lanes test 32 tiles at a time)
            const int32_t pmax = nrow_cta > 0 ? prm.row_pos[row_base + row0 + nrow_cta - 1] : -1;
            const int nft_total = (n_rows_req + kTileKeys - 1) / kTileKeys;
            const int32_t* kpc = prm.kpos_c + R[R_CBASE];
            for (int b = 0; b < nkt; b += 32)
                nct += __popc(__ballot_sync(0xffffffffu, b + lane < nkt && kpc[(b + lane) * kTileKeys] <= pmax));
            for (int b = 0; b < nft_total; b += 32)
                nft += __popc(__ballot_sync(0xffffffffu, b + lane < nft_total &&
                                                             prm.row_pos[row_base + (b + lane) * kTileKeys] <= pmax));
        }
        if (lane == 0) {
            misc[1] = nct;
            misc[2] = nft;
            misc[3] = t0;
            misc[4] = 0;
            const int n_all = nct + nft;
            const int ns = LSE ? 1 : PR[P_NSPLIT];
            const int sp = LSE ? 0 : chunk;
            misc[5] = (int)(((int64_t)sp * n_all) / ns);
            misc[6] = (int)(((int64_t)(sp + 1) * n_all) / ns);
        }
    }
    if (warp == kWarpMma) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), SM::kTmemCols);
        tmem_relinquish();
    }
    // (every K and V stage is filled by whole-tile copies: rows past a tensor's end read as 0)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);
    const int n_ct = misc[1], n_ft = misc[2], t0 = misc[3];
    const int n_tiles = n_ct + n_ft;
    const int jb = misc[5], n_loc = misc[6] - misc[5];   // tiles jb .. jb+n_loc-1 of the visible range

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ K producer
        // (The Q tiles were started by warp 0 during set-up.)  Per tile: lane l writes the
        // positions of keys l, l+32, l+64, l+96 (kNoPos for a missing key), fetched one tile ahead;
        // lane 0 then issues the rotated K tile.  The stage is reused once both Q K^T have read it
        // and both softmax groups have read its key positions.
        if (lane == 0) {
            prefetch_tmap(&tm_kcache);
            if (!LSE) prefetch_tmap(&tm_kfresh);
        }
        // logical position of key (lane + 32 r) of tile j (kNoPos if missing): LSE mode, every
        // cached token; attention, the compacted cached keys, then the fresh rows
        const int n_kept = n_pages * kPage - R[R_N_SEL];
        auto meta = [&](int j, int32_t (&pos)[4]) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int key = lane + 32 * r;
                pos[r] = kNoPos;
                if (j < n_ct) {
                    if (LSE) {
                        const int lp = (t0 + j) * kPagesPerTile + key / kPage;
                        if (lp < n_pages) pos[r] = page_pos[lp] + key % kPage;
                    } else {
                        const int ci = j * kTileKeys + key;
                        if (ci < n_kept) pos[r] = prm.kpos_c[R[R_CBASE] + ci];
                    }
                } else if (j < n_tiles) {
                    const int fr = (j - n_ct) * kTileKeys + key;
                    if (fr < n_rows_req) pos[r] = prm.row_pos[row_base + fr];
                }
            }
        };
        const int32_t kc_row0 = LSE ? kvh * L[L_TOTAL_TOKENS] + R[R_TOK_BASE] : kvh * L[L_TOTAL_VALID] + R[R_CBASE];
        int32_t pos_n[4];
        meta(jb, pos_n);
        int last[kKStages] = {-1, -1};
        for (int jj = 0; jj < n_loc; ++jj) {
            const int j = jb + jj, ks = jj & 1;
            int32_t pos[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) pos[r] = pos_n[r];
            meta(j + 1, pos_n);
            const bool ok = jj < kKStages ||
                            (mbar_wait(&bars[B_K_EMPTY + ks], ((jj >> 1) - 1) & 1, abort_flag) &&
                             mbar_wait(&bars[B_KPOS_FREE + ks], ((jj >> 1) - 1) & 1, abort_flag));
            if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll
            for (int r = 0; r < 4; ++r) sKpos(ks)[lane + 32 * r] = pos[r];
            uint64_t* full = &bars[B_K_FULL + ks];
            if (lane != 0) {
                mbar_arrive(full);
            } else {
                mbar_arrive_expect_tx(full, H * 16384);
                if (j < n_ct) {
                    const int32_t y = kc_row0 + (t0 + j) * kTileKeys;
                    for (int hb = 0; hb < H; ++hb) tma_load_2d(sKs(ks) + hb * 16384, &tm_kcache, full, hb * 64, y);
                } else {
                    const int32_t y = kvh * L[L_TOTAL_ROWS] + row_base + (j - n_ct) * kTileKeys;
                    for (int hb = 0; hb < H; ++hb) tma_load_2d(sKs(ks) + hb * 16384, &tm_kfresh, full, hb * 64, y);
                }
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
        if (!LSE && lane == 0) {
            prefetch_tmap(&tm_vcache);
            prefetch_tmap(&tm_vfresh);
            int last[kVStages] = {-1, -1};
            for (int jj = 0; jj < n_loc; ++jj) {
                const int j = jb + jj, vs = jj & 1;
                if (jj >= kVStages && !mbar_wait(&bars[B_V_EMPTY + vs], ((jj >> 1) - 1) & 1, abort_flag)) break;
                uint64_t* full = &bars[B_V_FULL + vs];
                mbar_arrive_expect_tx(full, H * 16384);
                if (j < n_ct) {
                    const int32_t y = kvh * L[L_TOTAL_VALID] + R[R_CBASE] + j * kTileKeys;
                    for (int hb = 0; hb < H; ++hb) tma_load_2d(sVs(vs) + hb * 16384, &tm_vcache, full, hb * 64, y);
                } else {
                    const int32_t fr = row_base + (j - n_ct) * kTileKeys;
                    for (int hb = 0; hb < H; ++hb)
                        tma_load_3d(sVs(vs) + hb * 16384, &tm_vfresh, full, hb * 64, kvh, fr);
                }
                last[vs] = jj;
            }
            for (int s2 = 0; s2 < kVStages; ++s2)
                if (last[s2] >= 0) mbar_drain(&bars[B_V_FULL + s2], (last[s2] >> 1) & 1);
        }
    } else if (warp == kWarpMma || warp == kWarpMmaB || warp == kWarpPvA || warp == kWarpPvB) {
        // ------------------------------------------------------------ MMA issuers
        const bool qk_role = warp == kWarpMma || warp == kWarpMmaB;
        const int t = (warp == kWarpMma || warp == kWarpPvA) ? 0 : 1;
        if (lane == 0) {
            const int nq = 2 * n_loc;   // halves of this CTA's key range
            bool ok = true;
            if (qk_role) {
                // Q K^T of half q = 2j + h of local key tile j: keys 64h .. 64h+63, S buffer q & 1
                constexpr uint32_t idesc_qk = idesc_f16(128, 64);
                const uint32_t aQ = smem_u32(sQ(t));
                auto issue_qk = [&](int q) {
                    const int j = q >> 1, h = q & 1;
                    const uint32_t aK = smem_u32(sKs(j & 1)) + h * 64 * 128;
                    const uint32_t tS = tmem + t * 128 + (q & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t a = desc_sw128_kmajor(aQ + (kk >> 2) * 16384 + (kk & 3) * 32);
                        const uint64_t b = desc_sw128_kmajor(aK + (kk >> 2) * 16384 + (kk & 3) * 32);
                        mma_bf16_ss(tS, a, b, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars[B_S_FULL + 2 * t + (q & 1)]);
                    if (h == 1) mma_commit(&bars[B_K_EMPTY + (j & 1)]);
                };
                ok = mbar_wait(&bars[B_Q_FULL], 0, abort_flag);
                ok = ok && (n_loc == 0 || mbar_wait(&bars[B_K_FULL + 0], 0, abort_flag));
                if (ok && n_loc > 0) {
                    tc_fence_after();
                    issue_qk(0);
                    issue_qk(1);
                }
                for (int q = 0; ok && q + 2 < nq; ++q) {
                    const int qn = q + 2, jn = qn >> 1;
                    // S(q+2) overwrites P(q): wait until P(q) V has read it (LSE mode: until the
                    // softmax has read S(q)); a new key tile must have landed first
                    ok = ((qn & 1) == 1 || mbar_wait(&bars[B_K_FULL + (jn & 1)], (jn >> 1) & 1, abort_flag)) &&
                         mbar_wait(&bars[(LSE ? B_P_FULL : B_PV_DONE) + 2 * t + (q & 1)], (q >> 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(qn);
                }
            } else if (!LSE) {
                // O += P(q) V(q): M=128, N=d in one instruction, K=64 keys in four steps
                constexpr uint32_t idesc_pv = idesc_bf16(128, D, true);
                const uint32_t tO = tmem + kTmemO + t * 128;
                for (int q = 0; ok && q < nq; ++q) {
                    const int j = q >> 1, h = q & 1;
                    ok = mbar_wait(&bars[B_P_FULL + 2 * t + (q & 1)], (q >> 1) & 1, abort_flag) &&
                         (h == 1 || mbar_wait(&bars[B_V_FULL + (j & 1)], (j >> 1) & 1, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t aV = smem_u32(sVs(j & 1)) + h * 64 * 128;
                    const uint32_t tP = tmem + t * 128 + (q & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < 64 / 16; ++kk)
                        mma_bf16_ts(tO, tP + kk * 8, desc_sw128_mn(aV + kk * 2048, 16384), idesc_pv,
                                    (q > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bars[B_PV_DONE + 2 * t + (q & 1)]);
                    if (q == nq - 1) mma_commit(&bars[B_O_DONE + t]);
                    if (h == 1) mma_commit(&bars[B_V_EMPTY + (j & 1)]);
                }
            }
            const int di = (qk_role ? 0 : 2) + t;
            mma_commit(&bars[B_DRAIN + di]);
            mbar_drain(&bars[B_DRAIN + di], 0);
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
        const uint32_t tO = tmem + lane_addr + kTmemO + t * 128;
        // output locations, fixed before the tile loop so that only one pointer stays live across it
        // (a split key range writes a normalized partial row plus its max and sum instead)
        __nv_bfloat16* out_row = nullptr;
        float2* ml_slot = nullptr;
        if (valid) {
            if (LSE) {
                ml_slot = prm.lse_part + R[R_LSE_BASE] +
                          ((int64_t)kvh * (R[R_N_QUERY] * g) + row * g + hl) * R[R_LSE_CHUNKS] + chunk;
            } else if (PR[P_NSPLIT] == 1) {
                out_row = prm.out + ((int64_t)(row_base + row) * Hq + kvh * g + hl) * D;
            } else {
                const int64_t prow = (int64_t)(PR[P_SLOT_BASE] + kvh * PR[P_NSPLIT] + chunk) *
                                         (kQTilesPerCta * kTileRows) + t * kTileRows + m;
                out_row = prm.part_o + prow * D;
                ml_slot = prm.part_ml + prow;
            }
        }
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int cut = 0;
        const int nq = 2 * n_loc;
        for (int q = 0; q < nq; ++q) {    // halves of the local key tiles
            const int j = q >> 1, h = q & 1, ks = j & 1;
            const uint32_t tS = tmem + lane_addr + t * 128 + (q & 1) * 64;
            ok = mbar_wait(&bars[B_S_FULL + 2 * t + (q & 1)], (q >> 1) & 1, abort_flag);
            if (h == 0) ok = ok && mbar_wait(&bars[B_K_FULL + ks], (j >> 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            if (h == 0) {
                // causal limit of this row inside the tile: keys are in increasing position order,
                // so the visible ones are a prefix (binary search)
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
            float mx;
            if (full) {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 64; e += 8) {
                    m4[0] = max3f(m4[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    m4[1] = max3f(m4[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                    m4[2] = max3f(m4[2], __uint_as_float(sv[e + 4]), __uint_as_float(sv[e + 5]));
                    m4[3] = max3f(m4[3], __uint_as_float(sv[e + 6]), __uint_as_float(sv[e + 7]));
                }
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            } else {
                // keys at or beyond the causal limit leave the row: score -inf
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (e >= cut_h) sv[e] = __float_as_uint(-INFINITY);
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 64; e += 8) {
                    m4[0] = max3f(m4[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    m4[1] = max3f(m4[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                    m4[2] = max3f(m4[2], __uint_as_float(sv[e + 4]), __uint_as_float(sv[e + 5]));
                    m4[3] = max3f(m4[3], __uint_as_float(sv[e + 6]), __uint_as_float(sv[e + 7]));
                }
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            const float m_new = fmaxf(m_run, mx);
            const bool need = m_new > m_run + 8.0f;     // lazy rescale: keep P <= 2^8
            const float alpha = need ? ex2(m_run - m_new) : 1.0f;
            if (need) { l_run *= alpha; m_run = m_new; }
            const float msub = m_run == -INFINITY ? 0.f : m_run;
            // p = 2^(s - m); P (bf16 pairs) goes over the half's first 32 S columns
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float p0 = ex2(__uint_as_float(sv[2 * e]) - msub);
                const float p1 = ex2(__uint_as_float(sv[2 * e + 1]) - msub);
                sum4[e & 3] += p0 + p1;
                pk[e] = pack_bf16x2(p0, p1);
            }
            if (!LSE) tmem_st32(tS, pk);
            l_run += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
            if (LSE) {
                tc_fence_before();
                mbar_arrive(&bars[B_P_FULL + 2 * t + (q & 1)]);
            } else {
                if (q > 0 && __any_sync(0xffffffffu, need)) {
                    // every earlier P V of this tile must be done before O is rescaled
                    ok = mbar_wait(&bars[B_PV_DONE + 2 * t + ((q - 1) & 1)], ((q - 1) >> 1) & 1, abort_flag);
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
                mbar_arrive(&bars[B_P_FULL + 2 * t + (q & 1)]);
            }
        }
        if (ml_slot != nullptr && ok) *ml_slot = make_float2(n_loc > 0 ? m_run : -INFINITY, l_run);
        if (LSE) {
            // The last key chunk of this (request, kv head, tile pair) to finish combines every row's
            // chunks, in chunk order, into the row's log2-sum-exp over all cached keys.
            const int chunks = R[R_LSE_CHUNKS];
            const int cidx = R[R_LSE_PAIR_BASE] + kvh * ((R[R_N_QUERY] * g + 2 * kTileRows - 1) / (2 * kTileRows)) + qpair;
            __threadfence();
            asm volatile("bar.sync 1, 256;" ::: "memory");   // the 256 softmax threads
            if (tid == 0) misc[7] = atomicAdd(prm.lse_count + cidx, 1) == chunks - 1 ? 1 : 0;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (misc[7]) {
                __threadfence();
                if (valid) {
                    const float2* ml = prm.lse_part + R[R_LSE_BASE] +
                                       ((int64_t)kvh * (R[R_N_QUERY] * g) + row * g + hl) * chunks;
                    // all chunks are loaded at once (chunks <= kMaxSplits), then combined in order
                    float2 v[kMaxSplits];
#pragma unroll
                    for (int c = 0; c < kMaxSplits; ++c) v[c] = c < chunks ? __ldcg(ml + c) : make_float2(-INFINITY, 0.f);
                    float M = -INFINITY;
#pragma unroll
                    for (int c = 0; c < kMaxSplits; ++c) M = fmaxf(M, v[c].x);
                    float S = 0.f;
#pragma unroll
                    for (int c = 0; c < kMaxSplits; ++c)
                        if (c < chunks) S += v[c].y * ex2(v[c].x - M);
                    prm.lse_final[((int64_t)kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE] + row) * g + hl] =
                        S > 0.f ? M + log2f(S) : INFINITY;
                }
                if (tid == 0) prm.lse_count[cidx] = 0;
            }
        }
        if (!LSE && ok && n_loc > 0) {
            ok = mbar_wait(&bars[B_O_DONE + t], 0, abort_flag);
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
