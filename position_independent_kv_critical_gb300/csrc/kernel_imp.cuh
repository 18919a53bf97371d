// Critical-layer importance, second pass (QCFuse, section 2B "Critical-layer attention
// profiling"; second summary, Phase 3: the query attends to the key cache of one layer only).
//
// imp[j] = sum_h sum_t exp2(s_{h,t,j} - lse2_{h,t}) with s in log2 units (the rotated query rows
// carry log2(e)/sqrt(d)) and lse2 the log2-sum-exp of row (h,t) over all cached keys of the request
// (from the first pass).  The tile is computed
// transposed, S^T = K_rot Q^T with M = 128 keys (TMEM lanes) and N = 256 query rows (columns), so
// that each thread owns one key and sums its own TMEM row -- no cross-thread reduction.  Both
// operands arrive rotated: the query rows, and the key tile from the call's rotated copy of the
// batch's cached keys (MiniPIC 2.1: rotation to the request's logical positions at use time).
// One CTA per (request, key tile, kv head); the per-kv-head partial sums are reduced in fixed
// head order by the last CTA of each key tile (deterministic).
#pragma once
#include "kernel_attn.cuh"

namespace pcf {

constexpr int kImpThreads = 192;
constexpr int kImpWarpMma = 4;
constexpr int kImpWarpTma = 5;
constexpr int kImpQRows = 256;

struct ImpParams {
    const int32_t* layout;
    const float2* lse_part;
    float* part;             // [Hkv][total_tokens]
    int32_t* counters;       // [total key tiles], zero on entry, left zero on exit
    float* importance;       // [total_tokens]
};

template <int D>
struct ImpSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kK = kTileKeys * D * 2;
    static constexpr int kQ = kImpQRows * D * 2;
    static constexpr int oK = 0;
    static constexpr int oQ = oK + kK;
    static constexpr int oLse = oQ + 2 * kQ;
    static constexpr int oBar = oLse + 2 * kImpQRows * 4;
    static constexpr int kNumBars = 12;
    static constexpr int oMisc = oBar + kNumBars * 8;
    static constexpr int kBytes = oMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
};

enum : int { I_K_FULL = 0, I_Q_FULL = 2 /*2*/, I_Q_EMPTY = 4 /*2*/, I_ACC_FULL = 6 /*2*/,
             I_ACC_FREE = 8 /*2*/, I_DRAIN = 10 };

__device__ __forceinline__ void named_sync_128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(kImpThreads, 1)
imp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kcache,
           const ImpParams prm) {
    using SM = ImpSmem<D>;
    constexpr int H = SM::kHalves;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem + SM::oK;
    auto sQs = [&](int b) { return smem + SM::oQ + b * SM::kQ; };
    auto sLse = [&](int b) { return reinterpret_cast<float*>(smem + SM::oLse) + b * kImpQRows; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::oBar);
    int32_t* misc = reinterpret_cast<int32_t*>(smem + SM::oMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* L = prm.layout;
    const int32_t* item = L + L[L_OFF_IMP] + kItemWords * blockIdx.x;
    const int req = item[0], t = item[1], kvh = item[2];
    const int32_t* R = L + L[L_OFF_REQ] + req * R_STRIDE;
    const int Hkv = L[L_HKV], g = L[L_GROUP];
    const int n_pages = R[R_N_PAGES];
    const int n_q = R[R_N_QUERY] * g;
    const int n_qc = (n_q + kImpQRows - 1) / kImpQRows;

    if (tid == 0) {
        mbar_init(&bars[I_K_FULL], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[I_Q_FULL + s], 1);
            mbar_init(&bars[I_Q_EMPTY + s], 1);
            mbar_init(&bars[I_ACC_FULL + s], 1);
            mbar_init(&bars[I_ACC_FREE + s], 128);
        }
        mbar_init(&bars[I_DRAIN], 1);
        fence_mbar_init();
        misc[4] = 0;
    }
    if (warp == kImpWarpMma) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), SM::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);

    if (warp == kImpWarpTma) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_kcache);
            // rotated key tile t of the request (rows past the request's keys are never summed)
            mbar_arrive_expect_tx(&bars[I_K_FULL], H * 16384);
            const int32_t ky = kvh * L[L_TOTAL_TOKENS] + R[R_TOK_BASE] + t * kTileKeys;
            for (int hb = 0; hb < H; ++hb)
                tma_load_2d(sK + hb * 16384, &tm_kcache, &bars[I_K_FULL], hb * 64, ky);

            const int32_t qy0 = (kvh * L[L_TOTAL_QUERY] + R[R_Q_BASE]) * g;
            int last[2] = {-1, -1};
            for (int qc = 0; qc < n_qc; ++qc) {
                const int b = qc & 1;
                if (qc >= 2 && !mbar_wait(&bars[I_Q_EMPTY + b], ((qc >> 1) - 1) & 1, abort_flag)) break;
                mbar_arrive_expect_tx(&bars[I_Q_FULL + b], H * kImpQRows * 128);
                for (int hb = 0; hb < H; ++hb)
                    tma_load_2d(sQs(b) + hb * kImpQRows * 128, &tm_q, &bars[I_Q_FULL + b], hb * 64,
                                qy0 + qc * kImpQRows);
                last[b] = qc;
            }
            mbar_drain(&bars[I_K_FULL], 0);
            for (int s = 0; s < 2; ++s)
                if (last[s] >= 0) mbar_drain(&bars[I_Q_FULL + s], (last[s] >> 1) & 1);
        }
    } else if (warp == kImpWarpMma) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(128, kImpQRows);
            const uint32_t aK = smem_u32(sK);
            bool ok = mbar_wait(&bars[I_K_FULL], 0, abort_flag);
            for (int qc = 0; ok && qc < n_qc; ++qc) {
                const int b = qc & 1;
                if (!mbar_wait(&bars[I_Q_FULL + b], (qc >> 1) & 1, abort_flag)) break;
                if (qc >= 2 && !mbar_wait(&bars[I_ACC_FREE + b], ((qc >> 1) - 1) & 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t aQ = smem_u32(sQs(b));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = desc_sw128_kmajor(aK + (kk >> 2) * 16384 + (kk & 3) * 32);
                    const uint64_t bq = desc_sw128_kmajor(aQ + (kk >> 2) * (kImpQRows * 128) + (kk & 3) * 32);
                    mma_bf16_ss(tmem + b * kImpQRows, a, bq, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars[I_ACC_FULL + b]);
                mma_commit(&bars[I_Q_EMPTY + b]);
            }
            mma_commit(&bars[I_DRAIN]);
            mbar_drain(&bars[I_DRAIN], 0);
        }
    } else {
        // warps 0-3: sum exp over the query rows for one key per thread
        bool ok = true;
        const int chunks = R[R_LSE_CHUNKS];
        const float2* part_in = prm.lse_part + R[R_LSE_BASE] + (int64_t)kvh * n_q * chunks;
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        float acc = 0.f;
        // every one of the 128 threads runs every iteration (named barriers inside): after an
        // abort the work is skipped, the barrier count stays the same
        for (int qc = 0; qc < n_qc; ++qc) {
            const int b = qc & 1;
            for (int rr = tid; rr < kImpQRows; rr += 128) {
                const int n = qc * kImpQRows + rr;
                float lse = INFINITY;
                if (n < n_q) {
                    float M = -INFINITY;
                    for (int cidx = 0; cidx < chunks; ++cidx) M = fmaxf(M, part_in[(int64_t)n * chunks + cidx].x);
                    float S = 0.f;
                    for (int cidx = 0; cidx < chunks; ++cidx) {
                        const float2 pl = part_in[(int64_t)n * chunks + cidx];
                        S += pl.y * ex2(pl.x - M);
                    }
                    lse = S > 0.f ? M + log2f(S) : INFINITY;
                }
                sLse(b)[rr] = lse;
            }
            named_sync_128();
            if (ok) ok = mbar_wait(&bars[I_ACC_FULL + b], (qc >> 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) continue;
            tc_fence_after();
            const int nvalid = min(kImpQRows, n_q - qc * kImpQRows);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sv[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    tmem_ld32(tmem + lane_addr + b * kImpQRows + half * 128 + cc * 32, sv[cc]);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int n = half * 128 + cc * 32 + e;
                        if (n < nvalid) acc += ex2(__uint_as_float(sv[cc][e]) - sLse(b)[n]);
                    }
            }
            tc_fence_before();
            mbar_arrive(&bars[I_ACC_FREE + b]);
        }
        // per-kv-head partial, then the last CTA of this key tile sums the heads in order
        const int total_tokens = L[L_TOTAL_TOKENS];
        const bool valid_key = (t * kPagesPerTile + tid / kPage) < n_pages;
        const int32_t tok = R[R_TOK_BASE] + t * kTileKeys + tid;
        if (ok && valid_key) prm.part[(int64_t)kvh * total_tokens + tok] = acc;
        __threadfence();
        named_sync_128();
        if (tid == 0) misc[5] = (atomicAdd(&prm.counters[R[R_KTILE_BASE] + t], 1) == Hkv - 1) ? 1 : 0;
        named_sync_128();
        if (misc[5]) {
            __threadfence();
            if (valid_key) {
                float s = 0.f;
                for (int h = 0; h < Hkv; ++h) s += __ldcg(prm.part + (int64_t)h * total_tokens + tok);
                prm.importance[tok] = s;
            }
            if (tid == 0) prm.counters[R[R_KTILE_BASE] + t] = 0;
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
