// Bandwidth-bound kernels of the hot path: rotation of per-request rows (query, fresh keys),
// per-span radix top-k and the row gather of the recompute batch.
#pragma once
#include "layout_format.h"
#include "ptx.cuh"

namespace pcf {

// ------------------------------------------------------------------ rope_rows
// Rotates rows (unrotated, bf16) at their logical positions and writes them in fp16 (the operand
// type of the Q K^T contractions), grouped by kv head for TMA:
// out[((h / gg) * n_rows + row) * gg + h % gg][D].  Used for the query rows (gg = Hq/Hkv, scaled
// by log2(e)/sqrt(d) so that Q K^T comes out in log2 units), the fresh keys (gg = 1) and, in page
// gather mode, the cached keys of every request: row r is the r-th cached token of the batch,
// read from the shared page blk[r / 16] at in-page offset r % 16 and rotated to the request's
// position page_pos[r / 16] + r % 16.  The pool itself is never written (MiniPIC 2.1: the shared
// blocks stay position-free); the rotated copy is per call, in the caller's workspace.
// With exclusion bits (the attention's copy), a token whose cached copy is replaced by a fresh
// row is left out: the others are compacted to row cidx[page] + (their rank among the page's
// kept tokens), their V rows are copied alongside and their positions recorded, so the attention
// streams only the keys that take part.
struct RopeJob {
    const __nv_bfloat16* x;  // rows [n_rows][heads][D], or the pool [n_phys][heads][16][D]
    const int32_t* pos;      // [n_rows] logical position of every row (row mode)
    __half* out;
    int32_t n_rows, heads, gg;
    float scale;             // folded into the output: log2(e)/sqrt(d) for queries, 1 for keys
    const int32_t* blk;      // page gather mode: physical page of every logical page (else null)
    const int32_t* page_pos; //   and the logical position of its first token
    int32_t n_phys;          //   pages in the pool
    const uint16_t* excl;    // compaction (page gather mode): exclusion bits per logical page, or null
    const int32_t* cidx;     //   compacted row of each page's first kept token
    const __nv_bfloat16* v_src;   // the V pool (same addressing as x)
    __nv_bfloat16* v_out;    //   V rows, [heads][n_out][D] like out
    int32_t* pos_out;        //   logical position of every compacted row
    int32_t n_out;           //   compacted rows
};

// The work is cut into tiles of 16 rows (one page in page gather mode) x up to 8 heads; a tile's
// bf16 rows and the cos/sin rows of its 16 positions are staged in shared memory by bulk copies
// (a page's heads are contiguous in the pool, so one copy each for K and V; a row's heads are
// contiguous in row mode, so one copy per row), on a ring of stages filled by one producer warp.
// The rotation reads shared memory only, so the bytes in flight per SM are set by the ring, not
// by registers: the per-row lookups (page, position, compacted row) are dependent loads, and a
// thread-per-row kernel that holds its data in registers runs out of warps to hide them with.
constexpr int kRopeRows = 16;            // rows of a tile
constexpr int kRopeHeads = 8;            // heads of a tile
// consumer warps: rotating keys alone is latency-bound and wants four per SM sub-partition; with
// the V rows copied too the stages are larger and two per sub-partition keep up (measured)
template <bool WITH_V>
__host__ __device__ constexpr int rope_consumer_warps() { return WITH_V ? 8 : 16; }
template <bool WITH_V>
__host__ __device__ constexpr int rope_threads() { return (rope_consumer_warps<WITH_V>() + 1) * 32; }   // + the producer warp

// A stage holds a tile's K rows (and V rows when the launch copies V) plus the cos/sin rows of its
// 16 positions; the ring takes as many stages as fit (the bytes in flight per SM are what keeps
// HBM busy: about one DRAM latency's worth of copy bandwidth, some 60 KB, beside the stage being
// rotated).
template <int D, bool WITH_V>
struct RopeSmem {
    static constexpr uint32_t kX = kRopeRows * kRopeHeads * D * 2;   // a tile's rows of K or V
    static constexpr uint32_t kCs = kRopeRows * D * 4;               // cos/sin of 16 positions
    static constexpr uint32_t kStage = (WITH_V ? 2 : 1) * kX + kCs;
    static constexpr int kStages = (int)((232448u - 1024u) / kStage) < 8 ? (int)((232448u - 1024u) / kStage) : 8;
    static constexpr uint32_t kMeta = kStages * kStage;              // int4 per stage
    static constexpr uint32_t kFull = kMeta + kStages * 16;          // mbarriers
    static constexpr uint32_t kEmpty = kFull + kStages * 8;
    static constexpr uint32_t kAbort = kEmpty + kStages * 8;
    static constexpr uint32_t kBytes = kAbort + 16;
    static_assert(kStages >= 2 && kBytes <= 232448, "rotation ring exceeds shared memory");
};

// A tile of one of the three jobs: rows [r0, r0 + nr), heads [h0, h0 + G).
struct RopeTile {
    int job;
    int32_t r0, nr, h0, G;
};
__device__ __forceinline__ RopeTile rope_tile(int64_t t, int64_t t_a, int64_t t_ab, const RopeJob& a,
                                              const RopeJob& b, const RopeJob& c3) {
    RopeTile T;
    T.job = t < t_a ? 0 : (t < t_ab ? 1 : 2);
    const RopeJob& J = T.job == 0 ? a : (T.job == 1 ? b : c3);
    const int64_t local = t - (T.job == 0 ? 0 : (T.job == 1 ? t_a : t_ab));
    const int ng = (J.heads + kRopeHeads - 1) / kRopeHeads;
    T.r0 = (int32_t)(local / ng) * kRopeRows;
    T.h0 = (int32_t)(local % ng) * kRopeHeads;
    T.nr = min(kRopeRows, J.n_rows - T.r0);
    T.G = min(kRopeHeads, J.heads - T.h0);
    return T;
}

// Persistent: CTA b takes tiles b, b + gridDim.x, ...  Tiles are numbered job by job; a job's
// tiles run row block by row block, head groups fastest (neighbouring tiles share cos/sin rows).
// WITH_V: some job of the launch copies V rows (the compacted cached keys); the others must not.
template <int D, bool WITH_V>
__global__ void __launch_bounds__(rope_threads<WITH_V>(), 1) rope_rows_kernel(RopeJob a, RopeJob b, RopeJob c3,
                                                                    const float2* __restrict__ rope, int32_t max_pos,
                                                                    int64_t t_a, int64_t t_ab, int64_t t_all,
                                                                    int32_t* __restrict__ zero, int32_t n_zero) {
    using SM = RopeSmem<D, WITH_V>;
    constexpr int kRopeStages = SM::kStages;
    constexpr int kRopeConsumerWarps = rope_consumer_warps<WITH_V>();
    constexpr int CPR = D / 16;   // 16-byte chunk pairs per head row
    extern __shared__ __align__(1024) uint8_t smem[];
    int4* s_meta = reinterpret_cast<int4*>(smem + SM::kMeta);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kFull);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + SM::kEmpty);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::kAbort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kRopeStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRopeConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    // counters of the kernels that follow, cleared here rather than by a separate memset
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < n_zero; i += (int64_t)gridDim.x * blockDim.x)
        zero[i] = 0;

    if (warp == kRopeConsumerWarps) {
        // ---------------- producer: metadata, then the bulk copies of the tile
        int64_t issued = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < t_all; t += gridDim.x, ++issued) {
            const int s = (int)(issued % kRopeStages);
            if (issued >= kRopeStages &&
                !mbar_wait(&empty[s], (uint32_t)((issued / kRopeStages - 1) & 1), abort_flag)) {
                ok = false;
                break;
            }
            const RopeTile T = rope_tile(t, t_a, t_ab, a, b, c3);
            const RopeJob& J = T.job == 0 ? a : (T.job == 1 ? b : c3);
            uint8_t* xs = smem + s * SM::kStage;
            uint8_t* vs = xs + SM::kX;
            uint8_t* cs = vs + (WITH_V ? SM::kX : 0);
            uint32_t valid = 0, ex = 0;
            int32_t ci = 0, pp = 0, ph = 0;
            if (J.blk != nullptr) {   // one page, all of its rows
                const int32_t page = T.r0 / kRopeRows;
                if (lane == 0) {
                    ph = J.blk[page];
                    pp = J.page_pos[page];
                    if (J.excl != nullptr) {
                        ex = J.excl[page];
                        ci = J.cidx[page];
                    }
                    if (ph < 0 || ph >= J.n_phys || pp < 0 || pp > max_pos - kRopeRows) {
                        set_dev_error(kDevErrBounds);
                    } else {
                        valid = (T.nr >= 32 ? 0xFFFFFFFFu : ((1u << T.nr) - 1u)) & ~ex;
                    }
                }
                valid = __shfl_sync(0xffffffffu, valid, 0);
                ph = __shfl_sync(0xffffffffu, ph, 0);
                pp = __shfl_sync(0xffffffffu, pp, 0);
                const uint32_t xb = (uint32_t)T.G * kRopeRows * D * 2;
                const bool with_v = WITH_V && J.v_src != nullptr;
                if (lane == 0) {
                    s_meta[s] = make_int4((int)valid, (int)ex, ci, pp);
                    mbar_arrive_expect_tx(&full[s], valid ? xb * (with_v ? 2u : 1u) + kRopeRows * D * 4 : 0u);
                }
                __syncwarp();
                if (valid) {
                    const int64_t off = ((int64_t)ph * J.heads + T.h0) * kRopeRows * D;
                    if (lane == 0) bulk_load(xs, J.x + off, xb, &full[s]);
                    if (lane == 1 && with_v) bulk_load(vs, J.v_src + off, xb, &full[s]);
                    if (lane == 2) bulk_load(cs, rope + (int64_t)pp * (D / 2), kRopeRows * D * 4, &full[s]);
                }
            } else {                   // 16 rows at their own positions
                int32_t p = 0;
                bool v = false;
                if (lane < T.nr) {
                    p = J.pos[T.r0 + lane];
                    v = p >= 0 && p < max_pos;
                    if (!v) set_dev_error(kDevErrBounds);
                }
                valid = __ballot_sync(0xffffffffu, v);
                const uint32_t rb = (uint32_t)T.G * D * 2;
                if (lane == 0) {
                    s_meta[s] = make_int4((int)valid, 0, 0, 0);
                    mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(valid) * (rb + D * 4));
                }
                __syncwarp();
                if (v) {
                    bulk_load(xs + lane * rb, J.x + ((int64_t)(T.r0 + lane) * J.heads + T.h0) * D, rb, &full[s]);
                    bulk_load(cs + lane * D * 4, rope + (int64_t)p * (D / 2), D * 4, &full[s]);
                }
            }
        }
        if (!ok) {   // an abort: let the copies still in flight land before the CTA exits
            if (lane == 0)
                for (int64_t j = issued > kRopeStages ? issued - kRopeStages : 0; j < issued; ++j)
                    mbar_drain(&full[j % kRopeStages], (uint32_t)((j / kRopeStages) & 1));
        }
        return;
    }

    // ---------------- consumers: rotate from shared memory, store fp16 (and the kept V rows)
    float big = 0.f;   // largest rotated magnitude: above fp16's range it is an error
    int64_t k = 0;
    for (int64_t t = blockIdx.x; t < t_all; t += gridDim.x, ++k) {
        const int s = (int)(k % kRopeStages);
        if (!mbar_wait(&full[s], (uint32_t)((k / kRopeStages) & 1), abort_flag)) break;
        const RopeTile T = rope_tile(t, t_a, t_ab, a, b, c3);
        const RopeJob& J = T.job == 0 ? a : (T.job == 1 ? b : c3);
        const int4 meta = s_meta[s];
        const uint32_t valid = (uint32_t)meta.x, ex = (uint32_t)meta.y;
        const uint8_t* xs = smem + s * SM::kStage;
        const uint8_t* vs = xs + SM::kX;
        const uint8_t* cs = vs + (WITH_V ? SM::kX : 0);
        const bool paged = J.blk != nullptr, compact = paged && J.excl != nullptr;
        const int32_t orow_n = compact ? J.n_out : J.n_rows;
        constexpr int kItems = kRopeRows * kRopeHeads * CPR;   // (row, head, chunk pair), chunk pairs fastest
        for (int it = tid; it < kItems; it += kRopeConsumerWarps * 32) {
            const int c = it % CPR, h = (it / CPR) % kRopeHeads, r = it / (CPR * kRopeHeads);
            if (h >= T.G || !((valid >> r) & 1u)) continue;
            int32_t oi = T.r0 + r;
            if (compact) {
                oi = meta.z + r - __popc(ex & ((1u << r) - 1u));   // kept tokens of the page before it
                if (oi < 0 || oi >= J.n_out) { set_dev_error(kDevErrBounds); continue; }
                if (c == 0 && T.h0 + h == 0) J.pos_out[oi] = meta.w + r;
            }
            const int idx = paged ? h * kRopeRows + r : r * T.G + h;
            const uint4 xa = *reinterpret_cast<const uint4*>(xs + idx * D * 2 + c * 16);
            const uint4 xb = *reinterpret_cast<const uint4*>(xs + idx * D * 2 + D + c * 16);
            const float4* cs4 = reinterpret_cast<const float4*>(cs + r * D * 4 + c * 64);
            const uint32_t ia[4] = {xa.x, xa.y, xa.z, xa.w};
            const uint32_t ib[4] = {xb.x, xb.y, xb.z, xb.w};
            uint32_t oa[4], ob[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 q = cs4[e];   // cos, sin of two consecutive frequencies
                const float a0 = bf16_lo(ia[e]) * J.scale, a1 = bf16_hi(ia[e]) * J.scale;
                const float b0 = bf16_lo(ib[e]) * J.scale, b1 = bf16_hi(ib[e]) * J.scale;
                oa[e] = pack_f16x2_track(fmaf(a0, q.x, -b0 * q.y), fmaf(a1, q.z, -b1 * q.w), big);
                ob[e] = pack_f16x2_track(fmaf(b0, q.x, a0 * q.y), fmaf(b1, q.z, a1 * q.w), big);
            }
            const int hh = T.h0 + h;
            const int64_t orow = ((int64_t)(hh / J.gg) * orow_n + oi) * J.gg + (hh % J.gg);
            __half* dst = J.out + orow * D;
            *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
            *reinterpret_cast<uint4*>(dst + D / 2 + 8 * c) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
            if (WITH_V && compact && J.v_src != nullptr) {   // the kept token's V row, unchanged
                __nv_bfloat16* vd = J.v_out + orow * D;
                *reinterpret_cast<uint4*>(vd + 8 * c) = *reinterpret_cast<const uint4*>(vs + idx * D * 2 + c * 16);
                *reinterpret_cast<uint4*>(vd + D / 2 + 8 * c) =
                    *reinterpret_cast<const uint4*>(vs + idx * D * 2 + D + c * 16);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!(big < kF16Limit)) set_dev_error(kDevErrRange);
}

// ------------------------------------------------------------------ block scan helper
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < NW ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < NW) s_warp[lane] = t;   // inclusive warp prefix
    }
    __syncthreads();
    const int before = (w > 0 ? s_warp[w - 1] : 0) + x - v;
    if (total) *total = s_warp[NW - 1];
    __syncthreads();
    return before;
}

// ------------------------------------------------------------------ per-span top-k
// QCFuse 2B: the Top-N tokens by critical-layer attention weight guide the recomputation; here
// N is taken per span (k_s), ties go to the lower index.  Radix select on the fp32 bit patterns
// (4 passes of 8 bits, shared-memory histograms), then two block scans in index order place the
// selected tokens in ascending order.  Blocks [0, n_spans) handle one span each; blocks
// [n_spans, n_spans + n_reqs) write the query rows' positions of one request each.
constexpr int kTopkThreads = 256;

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const int32_t* __restrict__ L,
                                                           const float* __restrict__ imp,
                                                           int32_t* __restrict__ sel_idx,
                                                           uint16_t* __restrict__ excl,
                                                           int32_t* __restrict__ row_pos) {
    extern __shared__ uint32_t s_bits[];   // selected-token bitmap of the span
    __shared__ int s_hist[256];
    __shared__ int s_warp[kTopkThreads / 32];
    __shared__ int s_bucket, s_above;
    // layout fields first: they do not depend on the previous kernel, which may still be running
    const int n_spans = L[L_N_SPANS];
    const int tid = threadIdx.x;
    if ((int)blockIdx.x >= n_spans) {
        const int b = blockIdx.x - n_spans;
        const int32_t* R = L + L[L_OFF_REQ] + b * R_STRIDE;
        const int32_t rb = R[R_ROW_BASE] + R[R_N_SEL], nq = R[R_N_QUERY], p0 = R[R_QUERY_POS0];
        grid_dep_wait();
        grid_dep_launch();
        for (int t = tid; t < nq; t += kTopkThreads) row_pos[rb + t] = p0 + t;
        return;
    }
    const int32_t* S = L + L[L_OFF_SPAN] + blockIdx.x * S_STRIDE;
    const int32_t* R = L + L[L_OFF_REQ] + S[S_REQ] * R_STRIDE;
    const int len = S[S_N_PAGES] * kPage;
    const int k = S[S_K];
    const int tok0 = S[S_PAGE_OFF] * kPage;              // request-local index of the span's first token
    const float* v = imp + R[R_TOK_BASE] + tok0;
    const int32_t sel_base = R[R_SEL_BASE] + S[S_SEL_OFF];
    const int32_t rrow = R[R_ROW_BASE] + S[S_SEL_OFF];
    const int32_t* ppos = L + L[L_OFF_PAGEPOS] + R[R_PAGE_BASE] + S[S_PAGE_OFF];
    uint16_t* ex = excl + R[R_PAGE_BASE] + S[S_PAGE_OFF];
    const int nwords = (len + 31) >> 5;
    for (int i = tid; i < nwords; i += kTopkThreads) s_bits[i] = 0u;
    grid_dep_wait();
    grid_dep_launch();

    uint32_t thr = 0;      // key of the k-th largest value
    int need_eq = 0;       // how many tokens equal to thr are taken (lowest indices first)
    if (k > 0 && k < len) {
        uint32_t prefix = 0, pmask = 0;
        int remaining = k;
        for (int shift = 24; shift >= 0; shift -= 8) {
            s_hist[tid] = 0;
            __syncthreads();
            for (int i = tid; i < len; i += kTopkThreads) {
                const uint32_t key = order_key(v[i]);
                if ((key & pmask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns buckets 255-8l .. 248-8l (descending)
                int cnt[8], tot = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) { cnt[q] = s_hist[255 - 8 * tid - q]; tot += cnt[q]; }
                int incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                const int excl_sum = incl - tot;
                const bool here = excl_sum < remaining && incl >= remaining;
                const unsigned m = __ballot_sync(0xffffffffu, here);
                if (here && tid == __ffs(m) - 1) {
                    int acc = excl_sum;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (acc + cnt[q] >= remaining) { s_bucket = 255 - 8 * tid - q; s_above = acc; break; }
                        acc += cnt[q];
                    }
                }
            }
            __syncthreads();
            const int bucket = s_bucket;
            remaining -= s_above;
            prefix |= (uint32_t)bucket << shift;
            pmask |= 255u << shift;
            __syncthreads();
        }
        thr = prefix;
        need_eq = remaining;
    }
    // contiguous index range per thread keeps index order in the scans
    const int per = (len + kTopkThreads - 1) / kTopkThreads;
    const int i0 = min(len, tid * per), i1 = min(len, i0 + per);
    int n_eq = 0;
    if (k > 0 && k < len)
        for (int i = i0; i < i1; ++i) n_eq += (order_key(v[i]) == thr);
    const int eq_before = block_excl_scan<kTopkThreads>(n_eq, s_warp, nullptr);
    int n_sel = 0;
    {
        int eq_rank = eq_before;
        for (int i = i0; i < i1; ++i) {
            bool take;
            if (k >= len) take = true;
            else if (k == 0) take = false;
            else {
                const uint32_t key = order_key(v[i]);
                take = key > thr || (key == thr && eq_rank < need_eq);
                eq_rank += (key == thr);
            }
            if (take) { ++n_sel; atomicOr(&s_bits[i >> 5], 1u << (i & 31)); }
        }
    }
    int total = 0;
    const int out_before = block_excl_scan<kTopkThreads>(n_sel, s_warp, &total);
    if (tid == 0 && total != k) set_dev_error(kDevErrBounds);
    int o = out_before;
    for (int i = i0; i < i1; ++i) {
        if ((s_bits[i >> 5] >> (i & 31)) & 1u) {
            if (o < k) {
                sel_idx[sel_base + o] = tok0 + i;
                row_pos[rrow + o] = ppos[i >> 4] + (i & 15);
            }
            ++o;
        }
    }
    __syncthreads();
    for (int p = tid; p < len / kPage; p += kTopkThreads)
        ex[p] = (uint16_t)((s_bits[p >> 1] >> ((p & 1) * 16)) & 0xFFFFu);
}

// ------------------------------------------------------------------ global Top-N
// QCFuse section 2B read literally: one Top-N over all of a request's cached tokens, with the
// request's budget N = sum of its spans' k (so the rows, their order and every buffer size stay
// those of the per-span selection).  One block per request: a radix select of the N-th largest
// key (fp32 bits, monotone for the non-negative importance and norms), then the tokens above it
// and the lowest-indexed ones equal to it, written in ascending order with the same outputs as
// topk_kernel; the block also writes the query rows' positions.
// The keys of one request sit in a narrow range (importance values share their sign and most of
// their exponent), so the select starts at the highest bit in which the request's smallest and
// largest keys differ and takes 11-bit digits (2048 bins) from there; a request of up to
// kTopnSmemKeys tokens keeps its keys in shared memory for all the passes.  Index order: warp w
// owns a contiguous segment of the request and walks it 32 tokens at a time (lane l on token
// base + l), so that loads are coalesced and shared-memory accesses conflict-free; ranks inside a
// warp come from ballots, the warps' starting ranks from a scan of their counts, and a ballot of
// the selected tokens is exactly one word of the bitmap.
constexpr int kTopnThreads = 1024;
constexpr int kTopnBins = 2048;
constexpr int kTopnDigit = 11;
constexpr int kTopnSmemKeys = 32768;

// dynamic shared memory: [bitmap of the largest request, in 16-byte groups][its keys, if staged]
__host__ __device__ inline size_t topn_smem_bytes(int max_tokens) {
    return (size_t)((max_tokens + 127) / 128) * 16 + (max_tokens <= kTopnSmemKeys ? (size_t)max_tokens * 4 : 0);
}

__global__ void __launch_bounds__(kTopnThreads) topn_global_kernel(const int32_t* __restrict__ L,
                                                                   const float* __restrict__ imp,
                                                                   int32_t* __restrict__ sel_idx,
                                                                   uint16_t* __restrict__ excl,
                                                                   int32_t* __restrict__ row_pos) {
    extern __shared__ __align__(16) uint32_t s_dyn[];
    __shared__ int s_hist[kTopnBins];
    __shared__ int s_warp[kTopnThreads / 32];
    __shared__ uint32_t s_red[2][kTopnThreads / 32];
    __shared__ int s_bucket, s_above;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // layout fields first: they do not depend on the previous kernel, which may still be running
    const int32_t* R = L + L[L_OFF_REQ] + blockIdx.x * R_STRIDE;
    const int len = R[R_N_PAGES] * kPage;
    const int k = R[R_N_SEL];
    const float* v = imp + R[R_TOK_BASE];
    const int32_t sel_base = R[R_SEL_BASE];
    const int32_t rrow = R[R_ROW_BASE];
    const int32_t* ppos = L + L[L_OFF_PAGEPOS] + R[R_PAGE_BASE];
    uint16_t* ex = excl + R[R_PAGE_BASE];
    const int nq = R[R_N_QUERY], p0 = R[R_QUERY_POS0];
    const int max_tok = L[L_MAX_TOKENS];
    uint32_t* s_bits = s_dyn;
    uint32_t* s_keys = s_dyn + ((max_tok + 127) / 128) * 4;   // the host sizes the allocation alike
    // staged when the largest request fits: the allocation follows that one
    const bool staged = max_tok <= kTopnSmemKeys;
    const bool partial = k > 0 && k < len;
    grid_dep_wait();
    grid_dep_launch();
    for (int t = tid; t < nq; t += kTopnThreads) row_pos[rrow + k + t] = p0 + t;

    // the keys (staged), and their smallest and largest
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    if (partial) {
        for (int i = tid; i < len; i += kTopnThreads) {
            const uint32_t key = order_key(v[i]);
            if (staged) s_keys[i] = key;
            kmin = min(kmin, key);
            kmax = max(kmax, key);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
            kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
        }
        if (lane == 0) { s_red[0][wid] = kmin; s_red[1][wid] = kmax; }
        __syncthreads();
        kmin = s_red[0][lane];
        kmax = s_red[1][lane];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
            kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
        }
    }
    auto key_at = [&](int i) { return staged ? s_keys[i] : order_key(v[i]); };

    uint32_t thr = 0;      // key of the k-th largest value
    int need_eq = 0;       // how many tokens equal to thr are taken (lowest indices first)
    if (partial) {
        if (kmin == kmax) {
            thr = kmax;
            need_eq = k;
        } else {
            const int hb = 31 - __clz(kmin ^ kmax);       // every key shares the bits above hb
            uint32_t pmask = hb == 31 ? 0u : ~((2u << hb) - 1u);
            uint32_t prefix = kmax & pmask;
            int remaining = k;
            for (int top = hb; top >= 0;) {
                const int w = min(kTopnDigit, top + 1), shift = top + 1 - w;
                const int nb = 1 << w;
                const uint32_t dmask = (uint32_t)nb - 1u;
                for (int b = tid; b < nb; b += kTopnThreads) s_hist[b] = 0;
                __syncthreads();
                for (int i = tid; i < len; i += kTopnThreads) {
                    const uint32_t key = key_at(i);
                    if ((key & pmask) == prefix) atomicAdd(&s_hist[(key >> shift) & dmask], 1);
                }
                __syncthreads();
                // bins in descending order, two per thread: the bucket holding the remaining-th
                // largest is where the count of larger keys first reaches it
                const int b_hi = nb - 1 - 2 * tid, b_lo = b_hi - 1;
                const int c_hi = b_hi >= 0 ? s_hist[b_hi] : 0, c_lo = b_lo >= 0 ? s_hist[b_lo] : 0;
                const int above = block_excl_scan<kTopnThreads>(c_hi + c_lo, s_warp, nullptr);
                if (above < remaining && above + c_hi + c_lo >= remaining) {
                    if (above + c_hi >= remaining) { s_bucket = b_hi; s_above = above; }
                    else { s_bucket = b_lo; s_above = above + c_hi; }
                }
                __syncthreads();
                prefix |= (uint32_t)s_bucket << shift;
                pmask |= dmask << shift;
                remaining -= s_above;
                top = shift - 1;
                __syncthreads();
            }
            thr = prefix;
            need_eq = remaining;
        }
    }

    // index order (see above): warp segments of 32-token groups
    constexpr int NW = kTopnThreads / 32;
    const int seg = ((len + NW * 32 - 1) / (NW * 32)) * 32;
    const int s0 = min(len, wid * seg), s1 = min(len, s0 + seg);
    const unsigned lt = (1u << lane) - 1u;
    auto scan_warps = [&](int cnt, int* total) {   // exclusive scan of one count per warp
        if (lane == 0) s_warp[wid] = cnt;
        __syncthreads();
        if (wid == 0) {
            int x = s_warp[lane];
            const int c = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            s_warp[lane] = x - c;
            if (lane == 31) s_above = x;
        }
        __syncthreads();
        const int before = s_warp[wid];
        if (total) *total = s_above;
        __syncthreads();
        return before;
    };
    // 1) tokens equal to the threshold before each warp's segment
    int eq_w = 0;
    if (partial)
        for (int b = s0; b < s1; b += 32) {
            const int i = b + lane;
            eq_w += __popc(__ballot_sync(0xffffffffu, i < s1 && key_at(i) == thr));
        }
    int eq_rank = scan_warps(eq_w, nullptr);
    // 2) the selection, as bitmap words
    int sel_w = 0;
    for (int b = s0; b < s1; b += 32) {
        const int i = b + lane;
        const bool valid = i < s1;
        const uint32_t key = (valid && partial) ? key_at(i) : 0u;
        const bool is_eq = valid && partial && key == thr;
        const unsigned eqm = __ballot_sync(0xffffffffu, is_eq);
        bool take;
        if (!valid || k == 0) take = false;
        else if (k >= len) take = true;
        else take = key > thr || (is_eq && eq_rank + __popc(eqm & lt) < need_eq);
        eq_rank += __popc(eqm);
        const unsigned tm = __ballot_sync(0xffffffffu, take);
        if (lane == 0) s_bits[b >> 5] = tm;
        sel_w += __popc(tm);
    }
    int total = 0;
    int o = scan_warps(sel_w, &total);
    if (tid == 0 && total != k) set_dev_error(kDevErrBounds);
    // 3) the selected tokens in ascending order, with their positions
    for (int b = s0; b < s1; b += 32) {
        const unsigned tm = s_bits[b >> 5];
        if ((tm >> lane) & 1u) {
            const int oo = o + __popc(tm & lt), i = b + lane;
            if (oo < k) {
                sel_idx[sel_base + oo] = i;
                row_pos[rrow + oo] = ppos[i >> 4] + (i & 15);
            }
        }
        o += __popc(tm);
    }
    __syncthreads();
    for (int p = tid; p < len / kPage; p += kTopnThreads)
        ex[p] = (uint16_t)((s_bits[p >> 1] >> ((p & 1) * 16)) & 0xFFFFu);
}

// ------------------------------------------------------------------ anchor key norms
// QCFuse section 2A / Phase 1: a cached token's key magnitude, read as the Euclidean norm of its
// unrotated key over every kv head and dimension (rotation preserves it, so positions do not
// matter).  One warp per token of the layout (global token t sits at in-page row t % 16 of
// logical page t / 16): lane l sums the squares of the 16-byte chunks l, l+32, ... of the
// token's Hkv x D values in fp32, a butterfly adds the lanes.  The pool is read before the
// dependency wait (no kernel writes it); the norms are written after it.
template <int D>
__global__ void __launch_bounds__(256) key_norm_kernel(const int32_t* __restrict__ L,
                                                       const __nv_bfloat16* __restrict__ k_pool,
                                                       float* __restrict__ norms) {
    constexpr int CPH = D / 8;   // 16-byte chunks per head row
    const int64_t tok = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int32_t total = L[L_TOTAL_TOKENS], hkv = L[L_HKV], n_phys = L[L_N_PHYS];
    float acc = 0.f;
    bool ok = true;
    if (tok < total) {
        const int32_t ph = L[L[L_OFF_BLOCK] + (int32_t)(tok / kPage)];
        ok = ph >= 0 && ph < n_phys;
        if (ok) {
            const __nv_bfloat16* base = k_pool + ((int64_t)ph * hkv * kPage + tok % kPage) * D;
            for (int q = lane; q < hkv * CPH; q += 32) {
                const int h = q / CPH, c = q % CPH;
                const uint4 x = *reinterpret_cast<const uint4*>(base + (int64_t)h * kPage * D + 8 * c);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
                    acc = fmaf(a, a, acc);
                    acc = fmaf(b, b, acc);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    grid_dep_wait();
    grid_dep_launch();
    if (tok < total && lane == 0) {
        if (!ok) set_dev_error(kDevErrBounds);
        else norms[tok] = sqrtf(acc);
    }
}

// ------------------------------------------------------------------ anchor pages
// QCFuse section 2A (injection): a request's anchors, selected per span in whole pages, are
// copied out of the shared pool into pages of their own, anchor i of the batch (in selection
// order) at page i / 16, row i % 16, every kv head, K and V alike; the fused attention then reads
// those pages as the prefix of the query.  One block per anchor page (its 16 anchors belong to
// one request because every request's anchor count is a multiple of 16): 16-byte chunks in
// destination order, so the stores are contiguous.
template <int D>
__global__ void __launch_bounds__(256) pack_anchor_kernel(const int32_t* __restrict__ L,
                                                          const int32_t* __restrict__ sel_idx,
                                                          const uint4* __restrict__ k_pool,
                                                          const uint4* __restrict__ v_pool,
                                                          uint4* __restrict__ k_anchor,
                                                          uint4* __restrict__ v_anchor) {
    constexpr int CPR = D / 8;   // 16-byte chunks per row
    const int32_t page = blockIdx.x;
    const int32_t first = page * kPage;   // first anchor of the page
    const int n_reqs = L[L_N_REQS], hkv = L[L_HKV], n_phys = L[L_N_PHYS];
    const int32_t* REQ = L + L[L_OFF_REQ];
    int lo = 0, hi = n_reqs - 1;   // last request with sel_base <= first
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (REQ[mid * R_STRIDE + R_SEL_BASE] <= first) lo = mid; else hi = mid - 1;
    }
    const int32_t* R = REQ + lo * R_STRIDE;
    const int32_t n_tok = R[R_N_PAGES] * kPage, tok_base = R[R_TOK_BASE];
    const int32_t* blk = L + L[L_OFF_BLOCK];
    grid_dep_wait();   // the anchors' indices come from the selection kernel
    grid_dep_launch();
    for (int q = threadIdx.x; q < hkv * kPage * CPR; q += blockDim.x) {
        const int h = q / (kPage * CPR), slot = (q / CPR) % kPage, c = q % CPR;
        const int32_t j = sel_idx[first + slot];
        if (j < 0 || j >= n_tok) { set_dev_error(kDevErrBounds); continue; }
        const int32_t t = tok_base + j;
        const int32_t ph = blk[t / kPage];
        if (ph < 0 || ph >= n_phys) { set_dev_error(kDevErrBounds); continue; }
        const int64_t src = (((int64_t)ph * hkv + h) * kPage + t % kPage) * CPR + c;
        const int64_t dst = (((int64_t)page * hkv + h) * kPage + slot) * CPR + c;
        k_anchor[dst] = k_pool[src];
        v_anchor[dst] = v_pool[src];
    }
}

// ------------------------------------------------------------------ row gather
// dst[sel_base_b + i] = src[tok_base_b + sel_idx[sel_base_b + i]] -- the inputs of the tokens
// chosen for recomputation (QCFuse Phase 4: discrete recomputation of the Top-N indices).
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ L,
                                                     const int32_t* __restrict__ sel_idx,
                                                     const uint4* __restrict__ src, int32_t row_chunks,
                                                     uint4* __restrict__ dst) {
    const int32_t r = blockIdx.x;
    const int n_reqs = L[L_N_REQS];
    const int32_t* REQ = L + L[L_OFF_REQ];
    int lo = 0, hi = n_reqs - 1;   // last request with sel_base <= r
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (REQ[mid * R_STRIDE + R_SEL_BASE] <= r) lo = mid; else hi = mid - 1;
    }
    const int32_t* R = REQ + lo * R_STRIDE;
    const int32_t n_tok = R[R_N_PAGES] * kPage, tok_base = R[R_TOK_BASE];
    // the layout search above does not depend on the previous kernel (which writes sel_idx)
    grid_dep_wait();
    grid_dep_launch();
    const int32_t j = sel_idx[r];
    if (j < 0 || j >= n_tok) {
        if (threadIdx.x == 0) set_dev_error(kDevErrBounds);
        return;
    }
    const uint4* s = src + (int64_t)(tok_base + j) * row_chunks;
    uint4* d = dst + (int64_t)r * row_chunks;
    for (int c = threadIdx.x; c < row_chunks; c += blockDim.x) d[c] = __ldg(s + c);
}

// ------------------------------------------------------------------ compaction scan
// Per logical page, the compacted row of its first cached token that takes part in the attention
// (exclusion bit clear): the request's base R_CBASE plus the kept tokens of the request's earlier
// pages.  One block per request.
constexpr int kScanThreads = 256;
__global__ void __launch_bounds__(kScanThreads) compact_scan_kernel(const int32_t* __restrict__ L,
                                                                    const uint16_t* __restrict__ excl,
                                                                    int32_t* __restrict__ cidx) {
    __shared__ int s_warp[kScanThreads / 32];
    const int32_t* R = L + L[L_OFF_REQ] + blockIdx.x * R_STRIDE;
    const int n_pages = R[R_N_PAGES], pb = R[R_PAGE_BASE];
    int carry = R[R_CBASE];
    grid_dep_wait();   // the exclusion bits come from the previous kernels
    grid_dep_launch();
    for (int p0 = 0; p0 < n_pages; p0 += kScanThreads) {
        const int p = p0 + threadIdx.x;
        const int kept = p < n_pages ? kPage - __popc((uint32_t)excl[pb + p]) : 0;
        int total;
        const int before = block_excl_scan<kScanThreads>(kept, s_warp, &total);
        if (p < n_pages) cidx[pb + p] = carry + before;
        carry += total;
    }
    // exclusion bits that do not leave exactly the request's kept count are a caller error
    if (threadIdx.x == 0 && carry != R[R_CBASE] + n_pages * kPage - R[R_N_SEL]) set_dev_error(kDevErrBounds);
}

// ------------------------------------------------------------------ split-range combine
// A (request, kv head, tile pair) whose key range was split over P_NSPLIT CTAs left, per split s,
// a normalized partial row O_s = (sum_u p_u v_u) / l_s together with (m_s, l_s) (running max in log2
// units, running sum).  The full row is sum_s w_s O_s / sum_s w_s with w_s = l_s 2^(m_s - max m),
// accumulated in one pass in split order (the running max rescales what was summed so far), so
// that the loads of several splits are in flight together.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const int32_t* __restrict__ L,
                                                      const __nv_bfloat16* __restrict__ part_o,
                                                      const float2* __restrict__ part_ml,
                                                      __nv_bfloat16* __restrict__ out) {
    constexpr int CH = D / 8;                   // 16-byte chunks per row
    constexpr int RPB = 256 / CH;               // rows per block
    const int32_t* item = L + L[L_OFF_COMB] + kItemWords * blockIdx.x;
    const int req = item[0], kvh = item[1], qpair = item[2];
    const int32_t* R = L + L[L_OFF_REQ] + req * R_STRIDE;
    const int32_t* PR = L + L[L_OFF_PAIR] + (R[R_PAIR_BASE] + qpair) * P_STRIDE;
    const int ns = PR[P_NSPLIT];
    const int g = L[L_GROUP], Hq = L[L_HQ];
    const int pr = blockIdx.y * RPB + threadIdx.x / CH;   // row within the pair, 0..255
    const int c = threadIdx.x % CH;
    const int tpt = kTileRows / g;
    const int tt = pr / kTileRows, mm = pr % kTileRows;
    const int row = qpair * kQTilesPerCta * tpt + tt * tpt + mm / g;
    const int32_t out_row = R[R_ROW_BASE] + row;
    const int64_t slot0 = (int64_t)PR[P_SLOT_BASE] + (int64_t)kvh * ns;
    const bool in_range = row < R[R_N_ROWS];
    // the layout fields above do not depend on the attention kernel, which may still be running
    grid_dep_wait();
    grid_dep_launch();
    if (!in_range) return;
    const int64_t stride = kQTilesPerCta * kTileRows;
    float M = -INFINITY, W = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int sp = 0; sp < ns; ++sp) {
        const float2 ml = part_ml[(slot0 + sp) * stride + pr];
        const uint4 v = *reinterpret_cast<const uint4*>(part_o + ((slot0 + sp) * stride + pr) * D + 8 * c);
        const bool live = ml.x != -INFINITY && ml.y > 0.f;
        const float m_new = live ? fmaxf(M, ml.x) : M;
        const float scale = m_new == M ? 1.f : ex2(M - m_new);
        const float w = live ? ml.y * ex2(ml.x - m_new) : 0.f;
        W = W * scale + w;
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[2 * e] = acc[2 * e] * scale + w * bf16_lo(u[e]);
            acc[2 * e + 1] = acc[2 * e + 1] * scale + w * bf16_hi(u[e]);
        }
        M = m_new;
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint4 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    const int hl = mm % g;
    *reinterpret_cast<uint4*>(out + ((int64_t)out_row * Hq + kvh * g + hl) * D + 8 * c) = o;
}

// ------------------------------------------------------------------ layer sum
// All-layer importance: out[j] = sum over l of per_layer[l][j], added in layer order (fp32,
// deterministic).  Four tokens per thread (16-byte loads); a tail of n % 4 tokens is done by the
// first threads one at a time.
__global__ void __launch_bounds__(256) layer_sum_kernel(const float* __restrict__ per_layer, int32_t n_layers,
                                                        int64_t n, float* __restrict__ out) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n4 = n / 4;
    if (gid < n4) {
        float4 acc = reinterpret_cast<const float4*>(per_layer)[gid];
        for (int l = 1; l < n_layers; ++l) {
            const float4 v = reinterpret_cast<const float4*>(per_layer + (int64_t)l * n)[gid];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4*>(out)[gid] = acc;
    } else if (gid - n4 < n - 4 * n4) {
        const int64_t j = 4 * n4 + (gid - n4);
        float acc = per_layer[j];
        for (int l = 1; l < n_layers; ++l) acc += per_layer[(int64_t)l * n + j];
        out[j] = acc;
    }
}

// ------------------------------------------------------------------ bounded-wait check
// Exercises the library's bounded mbarrier wait where it gives up: one thread initialises a
// barrier that expects one arrival, which never comes, and waits on it with a limit of `limit`
// clock cycles.  The wait runs out, raises the CTA's abort flag and the device error word
// (timeout), and the kernel returns: no copies, MMAs or tensor memory are involved, so there is
// nothing to drain.  Lane 0 records in flag[0] whether the wait returned false (1) or, against
// all expectation, true (2).
__global__ void __launch_bounds__(32) wait_limit_check_kernel(long long limit, int32_t* flag) {
    __shared__ uint64_t bar;
    __shared__ int abort_word;
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_word = 0;
        const bool done = mbar_wait(&bar, 0, reinterpret_cast<volatile int*>(&abort_word), limit);
        flag[0] = done ? 2 : 1;
    }
    __syncwarp();
}

}  // namespace pcf
