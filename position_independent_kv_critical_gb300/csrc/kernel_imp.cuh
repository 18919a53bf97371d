// Critical-layer importance, second pass (QCFuse, section 2B "Critical-layer attention
// profiling"; second summary, Phase 3: the query attends to the key cache of one layer only).
//
// imp[j] = sum_h sum_t exp2(s_{h,t,j} - lse2_{h,t}) with s in log2 units (the rotated query rows
// carry log2(e)/sqrt(d)) and lse2 the log2-sum-exp of row (h,t) over all cached keys of the request
// (written by the first pass).  Each tile is computed transposed, S^T = K_rot Q^T with M = 128
// keys (TMEM lanes) and N = 256 query rows (columns), so that each thread owns one key and sums
// its own TMEM row -- no cross-thread reduction.  The tensor core also subtracts the row's lse2: a
// last K=16 step multiplies a column pair of ones (key side) with (-lse2 rounded to fp16, the
// rounding remainder in fp16) on the query side, so S^T arrives as s - lse2 and each element costs
// one exponential and one add.  Both operands arrive rotated: the query rows, and
// the key tiles from the call's rotated copy of the batch's cached keys (MiniPIC 2.1: rotation to
// the request's logical positions at use time).
//
// One CTA per (request, run of key tiles, kv head, pair of 256-row query chunks).  Key tiles
// stream through a two-stage ring past the CTA's (at most two) query chunks, which stay in the two
// query buffers for the whole run, so each key tile is read once per CTA (a request with more
// than two chunks has one CTA per pair, neighbours in the work list that share the key tiles in
// L2); the S^T accumulator is double-buffered in TMEM, so the tensor core works on the next
// (tile, chunk) step while the exponentials of the current one run.  Each (chunk pair, query
// column half, kv head) writes its own partial sum per key; the last CTA of a run adds them in
// fixed order (chunk pairs, heads, halves: deterministic).
//   warps 0-7  exp-sum: warp w owns keys 32(w%4) .. +31 (its TMEM lane quarter) and the query
//              columns 128(w/4) .. +127 of every step
//   warp  8    TMEM allocation + single-thread tcgen05.mma issue
//   warp  9    TMA producer (key tiles, query chunks)
#pragma once
#include "kernel_attn.cuh"

namespace pcf {

constexpr int kImpThreads = 320;
// paged variant: two more warps (10, 11) rotate each key tile, copied from the pool pages, in place
constexpr int kImpThreadsPaged = 384;
constexpr int kImpWarpRot = 10;
template <bool PAGED> __host__ __device__ constexpr int imp_threads() { return PAGED ? kImpThreadsPaged : kImpThreads; }
constexpr int kImpExpThreads = 256;
constexpr int kImpWarpMma = 8;
constexpr int kImpWarpTma = 9;

struct ImpParams {
    const int32_t* layout;
    const float2* lse_part;  // pass 1: (max, sum) in log2 units, per request [kv head][chunk][row]
    float* part;             // [2][Hkv][total_tokens]: query column half, kv head, token
    int32_t* counters;       // [total key tiles], zero on entry, left zero on exit
    float* importance;       // [total_tokens]
    const float2* rope;      // paged: (cos, sin) table [max_pos][D/2]
};

template <int D>
struct ImpSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kK = kTileKeys * D * 2;
    static constexpr int kQ = kImpQRows * D * 2;
    static constexpr int oK = 0;                       // 2 key-tile stages
    static constexpr int oQ = oK + 2 * kK;             // 2 query-chunk buffers
    static constexpr int kSlabQ = kImpQRows * 16 * 2;  // [256][16] fp16: -lse2 (hi, lo) per row
    static constexpr int kSlabK = kTileKeys * 16 * 2;  // [128][16] fp16: ones in columns 0 and 1
    static constexpr int oQlse = oQ + 2 * kQ;          // 2 slabs (one per query-chunk buffer)
    static constexpr int oKones = oQlse + 2 * kSlabQ;
    static constexpr int oBar = oKones + kSlabK;
    static constexpr int kNumBars = 18;
    static constexpr int oMisc = oBar + kNumBars * 8;
    static constexpr int kBytes = oMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;         // 2 accumulators of 256 columns
};

enum : int { I_K_FULL = 0 /*2*/, I_K_EMPTY = 2 /*2*/, I_Q_FULL = 4 /*2*/, /* 6, 7 unused */
             I_ACC_FULL = 8 /*2*/, I_ACC_FREE = 10 /*2*/, I_LSE_FULL = 12 /*2*/, I_DRAIN = 14,
             I_KRAW_FULL = 16 /*2: paged, the key tile's page copies landed*/ };

__device__ __forceinline__ void named_sync_exp() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D, bool PAGED>
__global__ void __launch_bounds__(imp_threads<PAGED>(), 1)
imp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kcache,
           const ImpParams prm) {
    using SM = ImpSmem<D>;
    constexpr int H = SM::kHalves;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sKs = [&](int b) { return smem + SM::oK + b * SM::kK; };
    auto sQs = [&](int b) { return smem + SM::oQ + b * SM::kQ; };
    auto sQlse = [&](int b) { return smem + SM::oQlse + b * SM::kSlabQ; };
    uint8_t* sKones = smem + SM::oKones;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::oBar);
    int32_t* misc = reinterpret_cast<int32_t*>(smem + SM::oMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* L = prm.layout;
    const int32_t* item = L + L[L_OFF_IMP] + kItemWords * blockIdx.x;
    const int req = item[0], t0 = item[1], kvh = item[2] & 0xFFFF, cp = item[2] >> 16, nt = item[3];
    const int32_t* R = L + L[L_OFF_REQ] + req * R_STRIDE;
    const int Hkv = L[L_HKV], g = L[L_GROUP];
    const int n_pages = R[R_N_PAGES];
    const int n_q = R[R_N_QUERY] * g;
    const int n_cp = imp_chunk_pairs(R[R_N_QUERY], g);   // CTAs of this (run, kv head)
    const int qc0 = 2 * cp;                               // this CTA's first query chunk
    const int n_qc = max(0, min(2, (n_q + kImpQRows - 1) / kImpQRows - qc0));
    const int n_steps = nt * n_qc;
    // the (at most two) chunks stay in their own buffers, loaded once, and the steps go tile by
    // tile: step s = local tile s / n_qc, local chunk s % n_qc
    auto step_of = [&](int s, int& i, int& qc) { i = s / n_qc; qc = s - i * n_qc; };

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[I_K_FULL + b], PAGED ? 64 : 1);
            mbar_init(&bars[I_KRAW_FULL + b], 1);
            mbar_init(&bars[I_K_EMPTY + b], 1);
            mbar_init(&bars[I_Q_FULL + b], 1);
            mbar_init(&bars[I_ACC_FULL + b], 1);
            mbar_init(&bars[I_ACC_FREE + b], kImpExpThreads);
            mbar_init(&bars[I_LSE_FULL + b], kImpExpThreads);
        }
        mbar_init(&bars[I_DRAIN], 1);
        fence_mbar_init();
        misc[4] = 0;
    }
    // the previous kernel (row LSE, whose per-chunk max and sum are read here) may still be running
    // until this wait; the TMEM is taken only after it
    grid_dep_wait();
    grid_dep_launch();
    if (warp == kImpWarpMma) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), SM::kTmemCols);
        tmem_relinquish();
    }
    // the K=16 slabs start at zero; the key side gets its two columns of ones
    for (int i = tid; i < (2 * SM::kSlabQ + SM::kSlabK) / 16; i += imp_threads<PAGED>())
        reinterpret_cast<uint4*>(sQlse(0))[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid < kTileKeys) {
        *reinterpret_cast<__half*>(sKones + slab16_off(tid, 0)) = __float2half(1.0f);
        *reinterpret_cast<__half*>(sKones + slab16_off(tid, 1)) = __float2half(1.0f);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);

    if (warp == kImpWarpTma) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_kcache);
            const int32_t ky0 = kvh * L[L_TOTAL_TOKENS] + R[R_TOK_BASE] + t0 * kTileKeys;
            const int32_t qy0 = (kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE]) * g;
            const int32_t* blk = L + L[L_OFF_BLOCK] + R[R_PAGE_BASE];
            int lastk[2] = {-1, -1}, lastq[2] = {-1, -1};
            bool ok = true;
            // key tile t0 + i into stage kb: the rotated copy (one box per half) or, paged, its eight
            // pool pages (one 16-row box per page and half, a page past the request's last
            // repeating that last page), which the rotator warps then rotate in place
            auto load_k = [&](int kb, int i) {
                uint64_t* bar = &bars[(PAGED ? I_KRAW_FULL : I_K_FULL) + kb];
                mbar_arrive_expect_tx(bar, H * 16384);
                if (PAGED) {
                    for (int m = 0; m < kPagesPerTile; ++m) {
                        const int lp = min((t0 + i) * kPagesPerTile + m, n_pages - 1);
                        const int32_t y = (blk[lp] * Hkv + kvh) * kPage;
                        for (int hb = 0; hb < H; ++hb)
                            tma_load_2d(sKs(kb) + hb * 16384 + m * (kPage * 128), &tm_kcache, bar, hb * 64, y);
                    }
                } else {
                    for (int hb = 0; hb < H; ++hb)
                        tma_load_2d(sKs(kb) + hb * 16384, &tm_kcache, bar, hb * 64, ky0 + i * kTileKeys);
                }
            };
            // (a request without query rows has no steps: nothing is loaded)
            for (int i = 0; n_steps > 0 && ok && i < nt; ++i) {
                // rotated key tile t0 + i (rows past the request's keys are never summed)
                const int kb = i & 1;
                if (i >= 2 && !(ok = mbar_wait(&bars[I_K_EMPTY + kb], ((i >> 1) - 1) & 1, abort_flag))) break;
                load_k(kb, i);
                lastk[kb] = i;
                for (int qc = 0; i == 0 && qc < n_qc; ++qc) {   // each chunk once, into buffer qc
                    mbar_arrive_expect_tx(&bars[I_Q_FULL + qc], H * kImpQRows * 128);
                    for (int hb = 0; hb < H; ++hb)
                        tma_load_2d(sQs(qc) + hb * kImpQRows * 128, &tm_q, &bars[I_Q_FULL + qc], hb * 64,
                                    qy0 + (qc0 + qc) * kImpQRows);
                    lastq[qc] = 0;
                }
            }
            for (int b = 0; b < 2; ++b) {
                if (lastk[b] >= 0) mbar_drain(&bars[(PAGED ? I_KRAW_FULL : I_K_FULL) + b], (lastk[b] >> 1) & 1);
                if (lastq[b] >= 0) mbar_drain(&bars[I_Q_FULL + b], (lastq[b] >> 1) & 1);
            }
        }
    } else if (warp == kImpWarpMma) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(128, kImpQRows);
            bool ok = true;
            for (int s = 0; ok && s < n_steps; ++s) {
                int i, qc;
                step_of(s, i, qc);
                const int a = s & 1, qb = qc;
                // K stage: per tile in tile order; the chunks (and their -lse2 slabs) load once
                const int kidx = i;
                if (qc == 0) ok = mbar_wait(&bars[I_K_FULL + (kidx & 1)], (kidx >> 1) & 1, abort_flag);
                ok = ok && mbar_wait(&bars[I_Q_FULL + qb], 0, abort_flag) && mbar_wait(&bars[I_LSE_FULL + qb], 0, abort_flag);
                ok = ok && (s < 2 || mbar_wait(&bars[I_ACC_FREE + a], ((s >> 1) - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                // base descriptors plus constant step offsets: one thread then issues at the rate
                // shared memory allows, where descriptors rebuilt from the address each step do not
                const uint64_t dK = desc_sw128_kmajor(smem_u32(sKs(kidx & 1)));
                const uint64_t dQ = desc_sw128_kmajor(smem_u32(sQs(qb)));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tmem + a * kImpQRows, dK + sw128_k_step(kk), dQ + sw128_k_step(kk, kImpQRows * 128),
                                idesc, kk > 0 ? 1u : 0u);
                // + 1 * (-lse2_hi) + 1 * (-lse2_lo) per query row
                mma_bf16_ss(tmem + a * kImpQRows, desc_noswz_kmajor(smem_u32(sKones), 128, 256),
                            desc_noswz_kmajor(smem_u32(sQlse(qb)), 128, 256), idesc, 1u);
                mma_commit(&bars[I_ACC_FULL + a]);
                if (qc == n_qc - 1) mma_commit(&bars[I_K_EMPTY + (i & 1)]);
            }
            mma_commit(&bars[I_DRAIN]);
            mbar_drain(&bars[I_DRAIN], 0);
        }
    } else if (PAGED && warp >= kImpWarpRot) {
        // warps 10, 11 (paged): every key tile the producer copies from the pool pages is rotated in
        // place to the request's positions, in the producer's order, before the MMA reads it.
        // Thread t takes page t / 8 of the tile and 16-byte chunk pair c of 2*D/16 consecutive keys
        // (see rotate_page_keys); its table row is loaded one tile ahead.
        constexpr int CP = D / 16;
        constexpr int KPT = 2 * CP;
        const int rt = tid - kImpWarpRot * 32;
        const int m = rt / 8, c = rt % CP, r0 = ((rt % 8) / CP) * KPT;
        const int32_t* page_pos = L + L[L_OFF_PAGEPOS] + R[R_PAGE_BASE];
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
        const int n_loads = n_steps == 0 ? 0 : nt;   // each key tile once
        float4 tr[4];
        auto table_row = [&](int sidx) {
            const int i = sidx;
            const int lp = min((t0 + i) * kPagesPerTile + m, n_pages - 1);
            const float4* tp = reinterpret_cast<const float4*>(prm.rope + (int64_t)(page_pos[lp] + r0) * (D / 2) + 8 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e) tr[e] = tp[e];
        };
        if (n_loads > 0) table_row(0);
        for (int sidx = 0; sidx < n_loads; ++sidx) {
            const int kb = sidx & 1;
            const bool okr = mbar_wait(&bars[I_KRAW_FULL + kb], (sidx >> 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, okr)) break;
            uint64_t C[4], S[4], NS[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                C[e] = f2_pack(tr[e].x, tr[e].z);
                S[e] = f2_pack(tr[e].y, tr[e].w);
                NS[e] = f2_pack(-tr[e].y, -tr[e].w);
            }
            if (sidx + 1 < n_loads) table_row(sidx + 1);
            rotate_page_keys<D, KPT>(sKs(kb), kPage * m + r0, c, C, S, NS, STC, STS, NSTS);
            fence_proxy_async_smem();
            mbar_arrive(&bars[I_K_FULL + kb]);
        }
    } else {
        // warps 0-7: thread owns key `key` of every tile of the run, query columns ch*128 .. +127
        const int key = tid & 127, ch = tid >> 7;
        // pass 1's (max, sum) pairs of this kv head's query rows, one per key chunk
        const int chunks = R[R_LSE_CHUNKS];
        const float2* ml_g = prm.lse_part + R[R_LSE_BASE] + (int64_t)kvh * chunks * n_q;   // [chunk][row]
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int total_tokens = L[L_TOTAL_TOKENS];
        const int32_t tok_base = R[R_TOK_BASE];
        // -lse2 of the CTA's query chunk qc (0 or 1) into slab qc, as fp16 hi + lo (-30000 past the
        // last row: those columns contribute 0); thread tid writes row tid.  lse2 combines the row's
        // key chunks in chunk order: M = max of the maxima, lse2 = M + log2(sum_c s_c 2^(m_c - M)).
        auto prep = [&](int qc) {
            uint8_t* slab = sQlse(qc & 1);
            const int n = (qc0 + qc) * kImpQRows + tid;
            float v = -30000.f;
            if (n < n_q && chunks > 0) {
                float2 c2[kMaxSplits];
#pragma unroll
                for (int c = 0; c < kMaxSplits; ++c)
                    c2[c] = c < chunks ? __ldcg(ml_g + (int64_t)c * n_q + n) : make_float2(-INFINITY, 0.f);
                float M = -INFINITY;
#pragma unroll
                for (int c = 0; c < kMaxSplits; ++c) M = fmaxf(M, c2[c].x);
                float S = 0.f;
#pragma unroll
                for (int c = 0; c < kMaxSplits; ++c)
                    if (c < chunks) S += c2[c].y * ex2(c2[c].x - M);
                v = S > 0.f ? -(M + log2f(S)) : -INFINITY;
            }
            const __half hi = __float2half_rn(v);
            *reinterpret_cast<__half*>(slab + slab16_off(tid, 0)) = hi;
            *reinterpret_cast<__half*>(slab + slab16_off(tid, 1)) = __float2half_rn(v - __half2float(hi));
            fence_proxy_async_smem();
            mbar_arrive(&bars[I_LSE_FULL + (qc & 1)]);
        };
        if (n_steps > 0) prep(0);
        if (n_qc >= 2 && n_steps > 1) prep(1);
        bool ok = true;
        uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
        // this thread's (chunk pair, query column half, kv head) partial
        float* part_h = prm.part + ((int64_t)(cp * 2 + ch) * Hkv + kvh) * total_tokens;
        for (int s = 0; s < n_steps; ++s) {
            int i, qc;
            step_of(s, i, qc);
            const int a = s & 1;
            const int t = t0 + i;
            const bool valid_key = (t * kPagesPerTile + key / kPage) < n_pages;
            float* dst = part_h + tok_base + t * kTileKeys + key;
            if (ok) ok = mbar_wait(&bars[I_ACC_FULL + a], (s >> 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                uint32_t sv[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    tmem_ld32(tmem + lane_addr + a * kImpQRows + ch * 128 + cc * 32, sv[cc]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&bars[I_ACC_FREE + a]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        acc2[(e >> 1) & 1] = f2_add(acc2[(e >> 1) & 1], f2_pack(ex2(__uint_as_float(sv[cc][e])),
                                                                              ex2(__uint_as_float(sv[cc][e + 1]))));
            }
            if (qc == n_qc - 1) {   // the key's sum over the CTA's chunks
                float a0, a1, b0, b1;
                f2_unpack(acc2[0], a0, a1);
                f2_unpack(acc2[1], b0, b1);
                acc2[0] = acc2[1] = f2_pack(0.f, 0.f);
                if (ok && valid_key) *dst = (a0 + b0) + (a1 + b1);
            }
        }
        if (n_qc == 0)   // a request without query rows: every importance is 0
            for (int i = 0; i < nt; ++i)
                if (((t0 + i) * kPagesPerTile + key / kPage) < n_pages)
                    part_h[tok_base + (t0 + i) * kTileKeys + key] = 0.f;
        // the last of the run's Hkv * n_cp CTAs sums the chunk pairs and heads in order (the named
        // barriers order the partial writes before, and the reads after, thread 0's
        // acquire-release increment)
        named_sync_exp();
        const int cidx = R[R_KTILE_BASE] + t0;
        if (tid == 0) misc[5] = (atomic_add_acq_rel_gpu(&prm.counters[cidx], 1) == Hkv * n_cp - 1) ? 1 : 0;
        named_sync_exp();
        if (misc[5]) {
            for (int idx = tid; idx < nt * kTileKeys; idx += kImpExpThreads) {
                const int t = t0 + idx / kTileKeys, k = idx % kTileKeys;
                if ((t * kPagesPerTile + k / kPage) >= n_pages) continue;
                const int32_t tok = R[R_TOK_BASE] + t * kTileKeys + k;
                float sum = 0.f;
                for (int p = 0; p < n_cp; ++p)
                    for (int h = 0; h < Hkv; ++h)
                        sum += __ldcg(prm.part + ((int64_t)(2 * p) * Hkv + h) * total_tokens + tok) +
                               __ldcg(prm.part + ((int64_t)(2 * p + 1) * Hkv + h) * total_tokens + tok);
                prm.importance[tok] = sum;
            }
            if (tid == 0) prm.counters[cidx] = 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kImpWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, SM::kTmemCols);
    }
}

}  // namespace pcf
