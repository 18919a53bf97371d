// Device entry points of the C ABI (include/pcf.h): argument checks, TMA tensor maps, workspace
// carving and launches.  Every device buffer is the caller's; nothing here allocates.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/pcf.h"
#include "kernel_attn.cuh"
#include "kernel_imp.cuh"
#include "kernels_simple.cuh"
#include "layout_format.h"

using namespace pcf;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// Tensor maps are pure functions of their arguments; a small per-thread cache keeps the
// encoding off the per-call host path when a caller reuses its buffers from call to call.
struct MapKey {
    const void* base;
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    int32_t rank, dt;
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool valid;
};
thread_local MapEntry t_maps[16];
thread_local int t_maps_next = 0;

pcf_status encode_cached(CUtensorMap* m, const MapKey& k) {
    for (const MapEntry& e : t_maps)
        if (e.valid && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
            *m = e.map;
            return PCF_OK;
        }
    if (!get_encode()) return PCF_ERR_CUDA;
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, static_cast<CUtensorMapDataType>(k.dt), k.rank, const_cast<void*>(k.base), k.dims,
                          k.strides, k.box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PCF_ERR_CUDA;
    MapEntry& e = t_maps[t_maps_next];
    t_maps_next = (t_maps_next + 1) % 16;
    e.key = k;
    e.map = *m;
    e.valid = true;
    return PCF_OK;
}

// 2-D bf16 map over rows of `inner` elements (row stride `stride_bytes`), 128-byte swizzle,
// box = 64 elements x box_rows rows.  An empty tensor gives an all-zero (never used) map.
pcf_status make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_bytes,
                       uint32_t box_rows, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    std::memset(m, 0, sizeof(*m));
    if (rows == 0 || base == nullptr) return PCF_OK;
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = base;
    k.dims[0] = inner;
    k.dims[1] = rows;
    k.strides[0] = stride_bytes;
    k.box[0] = 64;
    k.box[1] = box_rows;
    k.rank = 2;
    k.dt = static_cast<int32_t>(dt);
    return encode_cached(m, k);
}

// 3-D map over [n2][n1][inner] (v_fresh: [rows][Hkv][D]), box = 64 x 1 x box2.
pcf_status make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t n1, uint64_t n2,
                       uint32_t box2) {
    std::memset(m, 0, sizeof(*m));
    if (n2 == 0 || base == nullptr) return PCF_OK;
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = base;
    k.dims[0] = inner;
    k.dims[1] = n1;
    k.dims[2] = n2;
    k.strides[0] = inner * 2;
    k.strides[1] = inner * n1 * 2;
    k.box[0] = 64;
    k.box[1] = 1;
    k.box[2] = box2;
    k.rank = 3;
    k.dt = static_cast<int32_t>(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    return encode_cached(m, k);
}

constexpr CUtensorMapDataType kF16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pcf_status check_layout(const pcf_layout* lay) {
    if (!lay || !lay->host || !lay->dev) return PCF_ERR_INVALID_ARG;
    const int32_t* H = lay->host;
    if (H[L_MAGIC] != kMagic || H[L_WORDS] < L_HEADER) return PCF_ERR_INVALID_ARG;
    if (H[L_D] != 64 && H[L_D] != 128) return PCF_ERR_UNSUPPORTED;
    return PCF_OK;
}

// sm_103 (GB300) must be the current device.  The answer and the device's SM count are kept per
// device ordinal: sms[dev] > 0 is the count of an sm_103 device, -1 marks another architecture.
std::atomic<int> g_dev_sms[256];

pcf_status check_device(int* n_sms = nullptr) {
    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PCF_ERR_NO_DEVICE;
    const bool cached = dev >= 0 && dev < 256;
    if (cached) {
        const int k = g_dev_sms[dev].load(std::memory_order_relaxed);
        if (k != 0) {
            if (k < 0) return PCF_ERR_NO_DEVICE;
            if (n_sms) *n_sms = k;
            return PCF_OK;
        }
    }
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return PCF_ERR_NO_DEVICE;
    const bool ok = major == 10 && minor == 3;
    if (cached) g_dev_sms[dev].store(ok ? sms : -1, std::memory_order_relaxed);
    if (!ok) return PCF_ERR_NO_DEVICE;
    if (n_sms) *n_sms = sms;
    return PCF_OK;
}

// the current device's SM count (after check_device succeeded on it)
int device_sms() {
    int n = kDefaultSms;
    check_device(&n);
    return n;
}

// Every kernel of the library is launched with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel in the stream is still running, set up what depends on no
// other kernel, and wait for that kernel in grid_dep_wait().  This hides most of the launch gap
// between the nine short kernels of a small batch.
template <typename... KArgs, typename... Args>
pcf_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? PCF_OK : PCF_ERR_CUDA;
}

size_t align_up(size_t x) { return (x + 1023) & ~size_t(1023); }

// rotated copy of every cached key of the batch: [Hkv][total_tokens][D] fp16
size_t kc_bytes(const int32_t* H) { return (size_t)H[L_HKV] * H[L_TOTAL_TOKENS] * H[L_D] * 2; }
// importance partials: [chunk pair][query column half][kv head][token]
size_t imp_part_floats(const int32_t* H) {
    return 2 * (size_t)imp_chunk_pairs(H[L_MAX_QUERY], H[L_GROUP]) * H[L_HKV] * H[L_TOTAL_TOKENS];
}

struct ScoreWs {
    size_t q, kc, lse, part, cnt, total;
};
ScoreWs score_ws(const int32_t* H) {
    ScoreWs w;
    w.q = 0;
    w.kc = align_up(w.q + (size_t)H[L_TOTAL_QUERY] * H[L_HQ] * H[L_D] * 2);
    w.lse = align_up(w.kc + kc_bytes(H));
    w.part = align_up(w.lse + (size_t)H[L_LSE_SLOTS] * sizeof(float2));
    // importance partials: per kv head and token, one per half of the query columns and pair of
    // query chunks
    w.cnt = align_up(w.part + imp_part_floats(H) * sizeof(float));
    // counters: importance runs (one per key tile at most) and the LSE kernel's item counter
    w.total = align_up(w.cnt + ((size_t)H[L_TOTAL_KTILES] + 1) * sizeof(int32_t));
    return w;
}

// The compacted attention's workspace: rotated fresh rows, and the rotated copy of the kept
// cached keys with their V rows and positions (it grows with the batch's cached tokens).
struct AttnWs {
    size_t q, k, kc, vc, kpos, cidx, po, pml, sched, total;
};
AttnWs attn_ws(const int32_t* H) {
    AttnWs w;
    const size_t valid_rows = (size_t)H[L_HKV] * H[L_TOTAL_VALID] * H[L_D];   // compacted K / V elements
    w.q = 0;
    w.k = align_up((size_t)H[L_TOTAL_ROWS] * H[L_HQ] * H[L_D] * 2);
    w.kc = align_up(w.k + (size_t)H[L_TOTAL_ROWS] * H[L_HKV] * H[L_D] * 2);
    w.vc = align_up(w.kc + valid_rows * 2);
    w.kpos = align_up(w.vc + valid_rows * 2);
    w.cidx = align_up(w.kpos + (size_t)H[L_TOTAL_VALID] * sizeof(int32_t));
    w.po = align_up(w.cidx + (size_t)H[L_TOTAL_PAGES] * sizeof(int32_t));
    const size_t prow = (size_t)H[L_ATTN_SLOTS] * kQTilesPerCta * kTileRows;   // partial rows
    w.pml = align_up(w.po + prow * H[L_D] * 2);
    w.sched = align_up(w.pml + prow * sizeof(float2));   // the attention kernel's item counter
    w.total = align_up(w.sched + sizeof(int32_t));
    return w;
}

// The paged attention's workspace grows with the batch's rows, not with its cached tokens: the
// cached keys and values are read from the pool pages by the attention kernel itself.
struct PagedWs {
    size_t q, k, cidx, po, pml, sched, total;
};
PagedWs paged_ws(const int32_t* H) {
    PagedWs w;
    w.q = 0;
    w.k = align_up((size_t)H[L_TOTAL_ROWS] * H[L_HQ] * H[L_D] * 2);
    w.cidx = align_up(w.k + (size_t)H[L_TOTAL_ROWS] * H[L_HKV] * H[L_D] * 2);
    w.po = align_up(w.cidx + (size_t)H[L_TOTAL_PAGES] * sizeof(int32_t));
    const size_t prow = (size_t)H[L_ATTN_SLOTS] * kQTilesPerCta * kTileRows;   // partial rows
    w.pml = align_up(w.po + prow * H[L_D] * 2);
    w.sched = align_up(w.pml + prow * sizeof(float2));   // the attention kernel's item counter
    w.total = align_up(w.sched + sizeof(int32_t));
    return w;
}

// the dynamic shared-memory limit of a kernel, per device: only ever raised (a launch with less
// than the limit is fine, so a kernel launched with several sizes keeps the largest)
std::mutex g_smem_mu;
std::map<std::pair<const void*, int>, int> g_smem_limit;
template <typename K>
pcf_status set_smem(K kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PCF_ERR_CUDA;
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    std::lock_guard<std::mutex> lock(g_smem_mu);
    auto it = g_smem_limit.find(key);
    if (it != g_smem_limit.end() && it->second >= bytes) return PCF_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return PCF_ERR_CUDA;
    g_smem_limit[key] = bytes;
    return PCF_OK;
}

// tiles of a RoPE job: 16-row blocks x groups of 8 heads
int64_t rope_tiles(const RopeJob& j) {
    if (!j.x || j.n_rows <= 0 || j.heads <= 0) return 0;
    return (int64_t)((j.n_rows + kRopeRows - 1) / kRopeRows) * ((j.heads + kRopeHeads - 1) / kRopeHeads);
}

template <int D>
pcf_status launch_rope(RopeJob a, RopeJob b, RopeJob c, const float2* rope, int32_t max_pos, cudaStream_t st,
                       int32_t* zero = nullptr, int32_t n_zero = 0) {
    // a job without rows takes no tiles
    if (!a.x || a.n_rows <= 0) a.x = nullptr;
    if (!b.x || b.n_rows <= 0) b.x = nullptr;
    if (!c.x || c.n_rows <= 0) c.x = nullptr;
    const int64_t t_a = rope_tiles(a), t_ab = t_a + rope_tiles(b), t_all = t_ab + rope_tiles(c);
    if (t_all == 0 && n_zero == 0) return PCF_OK;
    // persistent: one CTA per SM (the ring takes most of its shared memory), fewer for small jobs
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(t_all, device_sms()));
    const bool with_v = (a.x && a.v_src) || (b.x && b.v_src) || (c.x && c.v_src);
    auto go = [&](auto kernel, uint32_t bytes, int threads) -> pcf_status {
        pcf_status s = set_smem(kernel, (int)bytes);
        if (s != PCF_OK) return s;
        return launch(kernel, dim3((unsigned)blocks), dim3(threads), bytes, st, a, b, c, rope, max_pos, t_a, t_ab,
                      t_all, zero, n_zero);
    };
    return with_v ? go(rope_rows_kernel<D, true>, RopeSmem<D, true>::kBytes, rope_threads<true>())
                  : go(rope_rows_kernel<D, false>, RopeSmem<D, false>::kBytes, rope_threads<false>());
}

// the batch's cached keys, gathered from their pages and rotated to each request's positions
RopeJob cached_key_job(const pcf_layout* lay, const uint16_t* k_pool, __half* kc) {
    const int32_t* H = lay->host;
    return RopeJob{reinterpret_cast<const __nv_bfloat16*>(k_pool), nullptr, kc, H[L_TOTAL_TOKENS], H[L_HKV], 1, 1.f,
                   lay->dev + H[L_OFF_BLOCK], lay->dev + H[L_OFF_PAGEPOS], H[L_N_PHYS],
                   nullptr, nullptr, nullptr, nullptr, nullptr, 0};
}
// the cached keys that take part in the attention, compacted (rotated K, V copied, positions)
RopeJob kept_key_job(const pcf_layout* lay, const uint16_t* k_pool, const uint16_t* v_pool, const uint16_t* excl,
                     const int32_t* cidx, __half* kc, __nv_bfloat16* vc, int32_t* kpos) {
    RopeJob j = cached_key_job(lay, k_pool, kc);
    j.excl = excl;
    j.cidx = cidx;
    j.v_src = reinterpret_cast<const __nv_bfloat16*>(v_pool);
    j.v_out = vc;
    j.pos_out = kpos;
    j.n_out = lay->host[L_TOTAL_VALID];
    return j;
}

template <int D>
pcf_status score_impl(const pcf_layout* lay, const uint16_t* q_query, const uint16_t* k_pool, const float* rope,
                      float* importance, void* ws, cudaStream_t st) {
    const int32_t* H = lay->host;
    const ScoreWs w = score_ws(H);
    uint8_t* base = static_cast<uint8_t*>(ws);
    __half* q_rot = reinterpret_cast<__half*>(base + w.q);
    __half* kc = reinterpret_cast<__half*>(base + w.kc);
    float2* lse = reinterpret_cast<float2*>(base + w.lse);
    float* part = reinterpret_cast<float*>(base + w.part);
    int32_t* cnt = reinterpret_cast<int32_t*>(base + w.cnt);
    const int g = H[L_GROUP];
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    const float2* rope2 = reinterpret_cast<const float2*>(rope);

    const int32_t n_cnt = H[L_TOTAL_KTILES] + 1;   // cleared by the rotation kernel
    RopeJob qj{reinterpret_cast<const __nv_bfloat16*>(q_query), lay->dev + H[L_OFF_QPOS], q_rot, H[L_TOTAL_QUERY],
               H[L_HQ], g, scale_log2, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    RopeJob none{nullptr, nullptr, nullptr, 0, 0, 1, 1.f, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr,
                 nullptr, 0};
    pcf_status s = launch_rope<D>(qj, cached_key_job(lay, k_pool, kc), none, rope2, H[L_MAX_POS], st, cnt, n_cnt);
    if (s != PCF_OK) return s;

    CUtensorMap tq128, tq256, tkc, zero;
    std::memset(&zero, 0, sizeof(zero));
    const uint64_t qrows = (uint64_t)H[L_HKV] * H[L_TOTAL_QUERY] * g;
    if ((s = make_map_2d(&tq128, q_rot, D, qrows, D * 2, 128, kF16)) != PCF_OK) return s;
    if ((s = make_map_2d(&tq256, q_rot, D, qrows, D * 2, 256, kF16)) != PCF_OK) return s;
    if ((s = make_map_2d(&tkc, kc, D, (uint64_t)H[L_HKV] * H[L_TOTAL_TOKENS], D * 2, 128, kF16)) != PCF_OK)
        return s;

    if (H[L_N_LSE_ITEMS] > 0) {
        using SM = AttnSmem<D, true>;
        auto kern = attn_kernel<D, true, false>;
        if ((s = set_smem(kern, SM::kAlloc)) != PCF_OK) return s;
        AttnParams p{lay->dev, nullptr, nullptr, nullptr, lse, nullptr, nullptr, cnt + H[L_TOTAL_KTILES],
                     nullptr, nullptr, nullptr, nullptr, rope2};
        // persistent: at most one CTA per SM, items handed out in list order
        const int grid = std::min<int>(H[L_N_LSE_ITEMS], device_sms());
        if ((s = launch(kern, dim3(grid), dim3(attn_threads<false, true>()), SM::kAlloc, st, tq128, tkc, zero, zero, zero, zero, p)) !=
            PCF_OK)
            return s;
    }
    if (H[L_N_IMP_ITEMS] > 0) {
        using SM = ImpSmem<D>;
        auto kern = imp_kernel<D, false>;
        if ((s = set_smem(kern, SM::kAlloc)) != PCF_OK) return s;
        ImpParams p{lay->dev, lse, part, cnt, importance, rope2};
        if ((s = launch(kern, dim3(H[L_N_IMP_ITEMS]), dim3(kImpThreads), SM::kAlloc, st, tq256, tkc, p)) != PCF_OK)
            return s;
    }
    return PCF_OK;
}

// Paged scoring: the same two passes, reading the cached keys from their pool pages and rotating
// them inside the kernels (no copy of the cached keys).  Workspace: rotated query rows, the row
// LSE partials, the importance partials and the counters.
struct ScorePagedWs {
    size_t q, lse, part, cnt, total;
};
ScorePagedWs score_paged_ws(const int32_t* H) {
    ScorePagedWs w;
    w.q = 0;
    w.lse = align_up(w.q + (size_t)H[L_TOTAL_QUERY] * H[L_HQ] * H[L_D] * 2);
    w.part = align_up(w.lse + (size_t)H[L_LSE_SLOTS] * sizeof(float2));
    w.cnt = align_up(w.part + imp_part_floats(H) * sizeof(float));
    w.total = align_up(w.cnt + ((size_t)H[L_TOTAL_KTILES] + 1) * sizeof(int32_t));
    return w;
}

template <int D>
pcf_status score_paged_impl(const pcf_layout* lay, const uint16_t* q_query, const uint16_t* k_pool, const float* rope,
                            float* importance, void* ws, cudaStream_t st) {
    const int32_t* H = lay->host;
    const ScorePagedWs w = score_paged_ws(H);
    uint8_t* base = static_cast<uint8_t*>(ws);
    __half* q_rot = reinterpret_cast<__half*>(base + w.q);
    float2* lse = reinterpret_cast<float2*>(base + w.lse);
    float* part = reinterpret_cast<float*>(base + w.part);
    int32_t* cnt = reinterpret_cast<int32_t*>(base + w.cnt);
    const int g = H[L_GROUP];
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    const float2* rope2 = reinterpret_cast<const float2*>(rope);
    const int32_t n_cnt = H[L_TOTAL_KTILES] + 1;   // cleared by the rotation kernel
    RopeJob qj{reinterpret_cast<const __nv_bfloat16*>(q_query), lay->dev + H[L_OFF_QPOS], q_rot, H[L_TOTAL_QUERY],
               H[L_HQ], g, scale_log2, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    RopeJob none{nullptr, nullptr, nullptr, 0, 0, 1, 1.f, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr,
                 nullptr, 0};
    pcf_status s = launch_rope<D>(qj, none, none, rope2, H[L_MAX_POS], st, cnt, n_cnt);
    if (s != PCF_OK) return s;

    CUtensorMap tq128, tq256, tkp, zero;
    std::memset(&zero, 0, sizeof(zero));
    const uint64_t qrows = (uint64_t)H[L_HKV] * H[L_TOTAL_QUERY] * g;
    if ((s = make_map_2d(&tq128, q_rot, D, qrows, D * 2, 128, kF16)) != PCF_OK) return s;
    if ((s = make_map_2d(&tq256, q_rot, D, qrows, D * 2, 256, kF16)) != PCF_OK) return s;
    // the pool, unrotated and read only: one page (16 rows of one kv head) per copy
    if ((s = make_map_2d(&tkp, k_pool, D, (uint64_t)H[L_N_PHYS] * H[L_HKV] * kPage, D * 2, kPage)) != PCF_OK)
        return s;
    if (H[L_N_LSE_ITEMS] > 0) {
        using SM = AttnSmem<D, true, true>;
        auto kern = attn_kernel<D, true, true>;
        if ((s = set_smem(kern, SM::kAlloc)) != PCF_OK) return s;
        AttnParams p{lay->dev, nullptr, nullptr, nullptr, lse, nullptr, nullptr, cnt + H[L_TOTAL_KTILES],
                     nullptr, nullptr, nullptr, nullptr, rope2};
        const int grid = std::min<int>(H[L_N_LSE_ITEMS], device_sms());
        if ((s = launch(kern, dim3(grid), dim3(attn_threads<true, true>()), SM::kAlloc, st, tq128, tkp, zero, zero,
                        zero, zero, p)) != PCF_OK)
            return s;
    }
    if (H[L_N_IMP_ITEMS] > 0) {
        using SM = ImpSmem<D>;
        auto kern = imp_kernel<D, true>;
        if ((s = set_smem(kern, SM::kAlloc)) != PCF_OK) return s;
        ImpParams p{lay->dev, lse, part, cnt, importance, rope2};
        if ((s = launch(kern, dim3(H[L_N_IMP_ITEMS]), dim3(kImpThreadsPaged), SM::kAlloc, st, tq256, tkp, p)) !=
            PCF_OK)
            return s;
    }
    return PCF_OK;
}

template <int D>
pcf_status attention_impl(const pcf_layout* lay, const uint16_t* q_fresh, const uint16_t* k_fresh,
                          const uint16_t* v_fresh, const uint16_t* k_pool, const uint16_t* v_pool,
                          const uint16_t* excl, const int32_t* row_pos, const float* rope, uint16_t* out, void* ws,
                          cudaStream_t st, cudaEvent_t ev_start = nullptr, cudaEvent_t ev_stop = nullptr) {
    const int32_t* H = lay->host;
    if (H[L_N_ATTN_ITEMS] == 0) {   // no attention kernel: the timing events mark an empty span
        if (ev_start && cudaEventRecord(ev_start, st) != cudaSuccess) return PCF_ERR_CUDA;
        if (ev_stop && cudaEventRecord(ev_stop, st) != cudaSuccess) return PCF_ERR_CUDA;
        return PCF_OK;
    }
    const AttnWs w = attn_ws(H);
    uint8_t* base = static_cast<uint8_t*>(ws);
    __half* q_rot = reinterpret_cast<__half*>(base + w.q);
    __half* k_rot = reinterpret_cast<__half*>(base + w.k);
    __half* kc = reinterpret_cast<__half*>(base + w.kc);
    __nv_bfloat16* vc = reinterpret_cast<__nv_bfloat16*>(base + w.vc);
    int32_t* kpos_c = reinterpret_cast<int32_t*>(base + w.kpos);
    int32_t* cidx = reinterpret_cast<int32_t*>(base + w.cidx);
    const int g = H[L_GROUP];
    const float2* rope2 = reinterpret_cast<const float2*>(rope);
    const int32_t rows = H[L_TOTAL_ROWS];
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    RopeJob qj{reinterpret_cast<const __nv_bfloat16*>(q_fresh), row_pos, q_rot, rows, H[L_HQ], g, scale_log2,
               nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    RopeJob kj{reinterpret_cast<const __nv_bfloat16*>(k_fresh), row_pos, k_rot, rows, H[L_HKV], 1, 1.f,
               nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    pcf_status s;
    if (H[L_TOTAL_PAGES] > 0) {
        if ((s = launch(compact_scan_kernel, dim3(H[L_N_REQS]), dim3(kScanThreads), 0, st, lay->dev, excl, cidx)) !=
            PCF_OK)
            return s;
    }
    int32_t* sched = reinterpret_cast<int32_t*>(base + w.sched);
    s = launch_rope<D>(qj, kj, kept_key_job(lay, k_pool, v_pool, excl, cidx, kc, vc, kpos_c), rope2, H[L_MAX_POS], st,
                       sched, 1);
    if (s != PCF_OK) return s;

    CUtensorMap tq, tkc, tvc, tkf, tvf;
    if ((s = make_map_2d(&tq, q_rot, D, (uint64_t)H[L_HKV] * rows * g, D * 2, 128, kF16)) != PCF_OK) return s;
    // a batch without taking-part cached keys never reads these maps: point them at the fresh rows
    if (H[L_TOTAL_VALID] > 0) {
        const uint64_t vr = (uint64_t)H[L_HKV] * H[L_TOTAL_VALID];
        if ((s = make_map_2d(&tkc, kc, D, vr, D * 2, 128, kF16)) != PCF_OK) return s;
        if ((s = make_map_2d(&tvc, vc, D, vr, D * 2, 128)) != PCF_OK) return s;
    } else {
        if ((s = make_map_2d(&tkc, k_rot, D, (uint64_t)H[L_HKV] * rows, D * 2, 128, kF16)) != PCF_OK) return s;
        if ((s = make_map_2d(&tvc, v_fresh, D, (uint64_t)H[L_HKV] * rows, D * 2, 128)) != PCF_OK) return s;
    }
    if ((s = make_map_2d(&tkf, k_rot, D, (uint64_t)H[L_HKV] * rows, D * 2, 128, kF16)) != PCF_OK) return s;
    if ((s = make_map_3d(&tvf, v_fresh, D, H[L_HKV], rows, 128)) != PCF_OK) return s;

    using SM = AttnSmem<D, false, false>;
    auto kern = attn_kernel<D, false, false>;
    if ((s = set_smem(kern, SM::kAlloc)) != PCF_OK) return s;
    __nv_bfloat16* part_o = reinterpret_cast<__nv_bfloat16*>(base + w.po);
    float2* part_ml = reinterpret_cast<float2*>(base + w.pml);
    AttnParams p{lay->dev, kpos_c, row_pos, reinterpret_cast<__nv_bfloat16*>(out), nullptr, part_o, part_ml, sched,
                 nullptr, nullptr, nullptr, nullptr, rope2};
    // persistent: at most one CTA per SM, items handed out in list order (largest estimate first)
    const int grid = std::min<int>(H[L_N_ATTN_ITEMS], device_sms());
    if (ev_start && cudaEventRecord(ev_start, st) != cudaSuccess) return PCF_ERR_CUDA;
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof(unused));
    if ((s = launch(kern, dim3(grid), dim3(kAttnThreads), SM::kAlloc, st, tq, tkc, tvc, tkf, tvf, unused, p)) != PCF_OK)
        return s;
    if (ev_stop && cudaEventRecord(ev_stop, st) != cudaSuccess) return PCF_ERR_CUDA;
    if (H[L_N_COMB] > 0) {
        if ((s = launch(combine_kernel<D>, dim3(H[L_N_COMB], D / 8), dim3(256), 0, st, lay->dev,
                        (const __nv_bfloat16*)part_o, (const float2*)part_ml,
                        reinterpret_cast<__nv_bfloat16*>(out))) != PCF_OK)
            return s;
    }
    return PCF_OK;
}

template <int D>
pcf_status paged_attention_impl(const pcf_layout* lay, const uint16_t* q_fresh, const uint16_t* k_fresh,
                          const uint16_t* v_fresh, const uint16_t* k_pool, const uint16_t* v_pool,
                          const uint16_t* excl, const int32_t* row_pos, const float* rope, uint16_t* out, void* ws,
                          cudaStream_t st, cudaEvent_t ev_start = nullptr, cudaEvent_t ev_stop = nullptr) {
    const int32_t* H = lay->host;
    if (H[L_N_ATTN_ITEMS] == 0) {   // no attention kernel: the timing events mark an empty span
        if (ev_start && cudaEventRecord(ev_start, st) != cudaSuccess) return PCF_ERR_CUDA;
        if (ev_stop && cudaEventRecord(ev_stop, st) != cudaSuccess) return PCF_ERR_CUDA;
        return PCF_OK;
    }
    const PagedWs w = paged_ws(H);
    uint8_t* base = static_cast<uint8_t*>(ws);
    __half* q_rot = reinterpret_cast<__half*>(base + w.q);
    __half* k_rot = reinterpret_cast<__half*>(base + w.k);
    int32_t* cidx = reinterpret_cast<int32_t*>(base + w.cidx);
    const int g = H[L_GROUP];
    const float2* rope2 = reinterpret_cast<const float2*>(rope);
    const int32_t rows = H[L_TOTAL_ROWS];
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    RopeJob qj{reinterpret_cast<const __nv_bfloat16*>(q_fresh), row_pos, q_rot, rows, H[L_HQ], g, scale_log2,
               nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    RopeJob kj{reinterpret_cast<const __nv_bfloat16*>(k_fresh), row_pos, k_rot, rows, H[L_HKV], 1, 1.f,
               nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    RopeJob none{nullptr, nullptr, nullptr, 0, 0, 1, 1.f, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr,
                 nullptr, 0};
    pcf_status s;
    // per page, the request's kept tokens before it: a recomputed token's rank among the request's
    // recomputed rows follows from it, and the attention kernel puts that fresh row in its place
    if (H[L_TOTAL_PAGES] > 0) {
        if ((s = launch(compact_scan_kernel, dim3(H[L_N_REQS]), dim3(kScanThreads), 0, st, lay->dev, excl, cidx)) !=
            PCF_OK)
            return s;
    }
    int32_t* sched = reinterpret_cast<int32_t*>(base + w.sched);
    // the fresh rows (recomputed tokens and queries) are rotated once, at their row positions
    s = launch_rope<D>(qj, kj, none, rope2, H[L_MAX_POS], st, sched, 1);
    if (s != PCF_OK) return s;

    CUtensorMap tq, tkp, tvp, tkf, tvf;
    if ((s = make_map_2d(&tq, q_rot, D, (uint64_t)H[L_HKV] * rows * g, D * 2, 128, kF16)) != PCF_OK) return s;
    // the pool, unrotated and read only: one page (16 rows of one kv head) per copy.  A batch
    // without cached tokens never reads these maps: point them at the fresh rows.
    if (H[L_TOTAL_PAGES] > 0) {
        const uint64_t pr = (uint64_t)H[L_N_PHYS] * H[L_HKV] * kPage;
        if ((s = make_map_2d(&tkp, k_pool, D, pr, D * 2, kPage)) != PCF_OK) return s;
        if ((s = make_map_2d(&tvp, v_pool, D, pr, D * 2, kPage)) != PCF_OK) return s;
    } else {
        if ((s = make_map_2d(&tkp, k_fresh, D, (uint64_t)H[L_HKV] * rows, D * 2, kPage)) != PCF_OK) return s;
        if ((s = make_map_2d(&tvp, v_fresh, D, (uint64_t)H[L_HKV] * rows, D * 2, kPage)) != PCF_OK) return s;
    }
    if ((s = make_map_2d(&tkf, k_rot, D, (uint64_t)H[L_HKV] * rows, D * 2, 128, kF16)) != PCF_OK) return s;
    if ((s = make_map_3d(&tvf, v_fresh, D, H[L_HKV], rows, 128)) != PCF_OK) return s;
    // the fresh keys of a cached tile's recomputed tokens, staged with the tile
    CUtensorMap tks;
    if ((s = make_map_2d(&tks, k_rot, D, (uint64_t)H[L_HKV] * rows, D * 2, kStageRows, kF16)) != PCF_OK) return s;

    using SM = AttnSmem<D, false, true>;
    auto kern = attn_kernel<D, false, true>;
    if ((s = set_smem(kern, SM::kAlloc)) != PCF_OK) return s;
    __nv_bfloat16* part_o = reinterpret_cast<__nv_bfloat16*>(base + w.po);
    float2* part_ml = reinterpret_cast<float2*>(base + w.pml);
    AttnParams p{lay->dev, nullptr, row_pos, reinterpret_cast<__nv_bfloat16*>(out), nullptr, part_o, part_ml, sched,
                 excl, cidx, k_rot, reinterpret_cast<const __nv_bfloat16*>(v_fresh), rope2};
    // persistent: at most one CTA per SM, items handed out in list order (largest estimate first)
    const int grid = std::min<int>(H[L_N_ATTN_ITEMS], device_sms());
    if (ev_start && cudaEventRecord(ev_start, st) != cudaSuccess) return PCF_ERR_CUDA;
    if ((s = launch(kern, dim3(grid), dim3(kAttnThreadsPaged), SM::kAlloc, st, tq, tkp, tvp, tkf, tvf, tks, p)) !=
        PCF_OK)
        return s;
    if (ev_stop && cudaEventRecord(ev_stop, st) != cudaSuccess) return PCF_ERR_CUDA;
    if (H[L_N_COMB] > 0) {
        if ((s = launch(combine_kernel<D>, dim3(H[L_N_COMB], D / 8), dim3(256), 0, st, lay->dev,
                        (const __nv_bfloat16*)part_o, (const float2*)part_ml,
                        reinterpret_cast<__nv_bfloat16*>(out))) != PCF_OK)
            return s;
    }
    return PCF_OK;
}

}  // namespace

extern "C" pcf_status pcf_score_workspace_bytes(const int32_t* layout_host, size_t* bytes) {
    if (!layout_host || !bytes || layout_host[L_MAGIC] != kMagic) return PCF_ERR_INVALID_ARG;
    *bytes = score_ws(layout_host).total;
    return PCF_OK;
}

extern "C" pcf_status pcf_attention_workspace_bytes(const int32_t* layout_host, size_t* bytes) {
    if (!layout_host || !bytes || layout_host[L_MAGIC] != kMagic) return PCF_ERR_INVALID_ARG;
    *bytes = attn_ws(layout_host).total;
    return PCF_OK;
}

extern "C" pcf_status pcf_attention_paged_workspace_bytes(const int32_t* layout_host, size_t* bytes) {
    if (!layout_host || !bytes || layout_host[L_MAGIC] != kMagic) return PCF_ERR_INVALID_ARG;
    *bytes = paged_ws(layout_host).total;
    return PCF_OK;
}

extern "C" pcf_status pcf_score(const pcf_layout* layout, const uint16_t* q_query, const uint16_t* k_pool,
                                const float* rope, float* importance, void* ws, size_t ws_bytes, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (H[L_TOTAL_TOKENS] == 0) return PCF_OK;
    if (!k_pool || !rope || !importance || !ws || (H[L_TOTAL_QUERY] > 0 && !q_query)) return PCF_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(rope) || !aligned16(ws) || (q_query && !aligned16(q_query)))
        return PCF_ERR_INVALID_ARG;
    if (ws_bytes < score_ws(H).total) return PCF_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_device()) != PCF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return H[L_D] == 128 ? score_impl<128>(layout, q_query, k_pool, rope, importance, ws, st)
                         : score_impl<64>(layout, q_query, k_pool, rope, importance, ws, st);
}

extern "C" pcf_status pcf_score_layers(const pcf_layout* layout, int32_t n_layers,
                                       const uint16_t* const* q_query_layers, const uint16_t* const* k_pool_layers,
                                       const float* rope, float* importance_layers, float* importance_sum, void* ws,
                                       size_t ws_bytes, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (n_layers < 1 || n_layers > 4096 || !q_query_layers || !k_pool_layers) return PCF_ERR_INVALID_ARG;
    if (H[L_TOTAL_TOKENS] == 0) return PCF_OK;
    if (!rope || !importance_layers || !importance_sum || !ws) return PCF_ERR_INVALID_ARG;
    if (!aligned16(rope) || !aligned16(ws) || !aligned16(importance_layers) || !aligned16(importance_sum))
        return PCF_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        const uint16_t* q = q_query_layers[l];
        const uint16_t* k = k_pool_layers[l];
        if (!k || !aligned16(k) || (H[L_TOTAL_QUERY] > 0 && (!q || !aligned16(q)))) return PCF_ERR_INVALID_ARG;
    }
    if (ws_bytes < score_ws(H).total) return PCF_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_device()) != PCF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t n = H[L_TOTAL_TOKENS];
    // layer by layer on the stream (the workspace is reused: each layer's kernels start after the
    // previous layer's have finished with it)
    for (int l = 0; l < n_layers; ++l) {
        float* imp = importance_layers + (int64_t)l * n;
        s = H[L_D] == 128 ? score_impl<128>(layout, q_query_layers[l], k_pool_layers[l], rope, imp, ws, st)
                          : score_impl<64>(layout, q_query_layers[l], k_pool_layers[l], rope, imp, ws, st);
        if (s != PCF_OK) return s;
    }
    const int64_t threads = n / 4 + n % 4;
    return launch(layer_sum_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st,
                  (const float*)importance_layers, n_layers, n, importance_sum);
}

extern "C" pcf_status pcf_score_paged_workspace_bytes(const int32_t* layout_host, size_t* bytes) {
    if (!layout_host || !bytes || layout_host[L_MAGIC] != kMagic) return PCF_ERR_INVALID_ARG;
    *bytes = score_paged_ws(layout_host).total;
    return PCF_OK;
}

extern "C" pcf_status pcf_score_paged(const pcf_layout* layout, const uint16_t* q_query, const uint16_t* k_pool,
                                      const float* rope, float* importance, void* ws, size_t ws_bytes, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (H[L_TOTAL_TOKENS] == 0) return PCF_OK;
    if (!k_pool || !rope || !importance || !ws || (H[L_TOTAL_QUERY] > 0 && !q_query)) return PCF_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(rope) || !aligned16(ws) || (q_query && !aligned16(q_query)))
        return PCF_ERR_INVALID_ARG;
    if (ws_bytes < score_paged_ws(H).total) return PCF_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_device()) != PCF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return H[L_D] == 128 ? score_paged_impl<128>(layout, q_query, k_pool, rope, importance, ws, st)
                         : score_paged_impl<64>(layout, q_query, k_pool, rope, importance, ws, st);
}

extern "C" pcf_status pcf_select_topk(const pcf_layout* layout, const float* importance, int32_t* sel_idx,
                                      uint16_t* excl, int32_t* row_pos, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if ((H[L_TOTAL_TOKENS] > 0 && (!importance || !excl)) || (H[L_TOTAL_SEL] > 0 && !sel_idx) ||
        (H[L_TOTAL_ROWS] > 0 && !row_pos))
        return PCF_ERR_INVALID_ARG;
    if ((s = check_device()) != PCF_OK) return s;
    const int blocks = H[L_N_SPANS] + H[L_N_REQS];
    const int words = (H[L_MAX_SPAN_LEN] + 31) / 32;
    if (words * 4 > 48 * 1024) return PCF_ERR_UNSUPPORTED;
    return launch(topk_kernel, dim3(blocks), dim3(kTopkThreads), words * 4, static_cast<cudaStream_t>(stream),
                  layout->dev, importance, sel_idx, excl, row_pos);
}

extern "C" pcf_status pcf_select_topn_global(const pcf_layout* layout, const float* importance, int32_t* sel_idx,
                                             uint16_t* excl, int32_t* row_pos, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if ((H[L_TOTAL_TOKENS] > 0 && (!importance || !excl)) || (H[L_TOTAL_SEL] > 0 && !sel_idx) ||
        (H[L_TOTAL_ROWS] > 0 && !row_pos))
        return PCF_ERR_INVALID_ARG;
    if (H[L_N_REQS] == 0) return PCF_OK;
    if ((s = check_device()) != PCF_OK) return s;
    const int words = (H[L_MAX_TOKENS] + 31) / 32;
    if (words * 4 > 48 * 1024) return PCF_ERR_UNSUPPORTED;
    const size_t smem = topn_smem_bytes(H[L_MAX_TOKENS]);   // bitmap, then the keys when they fit
    if ((s = set_smem(topn_global_kernel, (int)smem)) != PCF_OK) return s;
    return launch(topn_global_kernel, dim3(H[L_N_REQS]), dim3(kTopnThreads), smem,
                  static_cast<cudaStream_t>(stream), layout->dev, importance, sel_idx, excl, row_pos);
}

extern "C" pcf_status pcf_key_norms(const pcf_layout* layout, const uint16_t* k_pool, float* norms, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (H[L_TOTAL_TOKENS] == 0) return PCF_OK;
    if (!k_pool || !norms || !aligned16(k_pool)) return PCF_ERR_INVALID_ARG;
    if ((s = check_device()) != PCF_OK) return s;
    const int64_t blocks = ((int64_t)H[L_TOTAL_TOKENS] * 32 + 255) / 256;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto* kp = reinterpret_cast<const __nv_bfloat16*>(k_pool);
    return H[L_D] == 128 ? launch(key_norm_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, st, layout->dev, kp, norms)
                         : launch(key_norm_kernel<64>, dim3((unsigned)blocks), dim3(256), 0, st, layout->dev, kp, norms);
}

extern "C" pcf_status pcf_pack_anchor_pages(const pcf_layout* layout, const int32_t* sel_idx, const uint16_t* k_pool,
                                            const uint16_t* v_pool, uint16_t* k_anchor, uint16_t* v_anchor,
                                            void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    // every request's anchors must fill whole pages
    for (int b = 0; b < H[L_N_REQS]; ++b)
        if (H[H[L_OFF_REQ] + b * R_STRIDE + R_N_SEL] % kPage != 0) return PCF_ERR_INVALID_ARG;
    if (H[L_TOTAL_SEL] == 0) return PCF_OK;
    if (!sel_idx || !k_pool || !v_pool || !k_anchor || !v_anchor) return PCF_ERR_INVALID_ARG;
    for (const void* p : {(const void*)k_pool, (const void*)v_pool, (const void*)k_anchor, (const void*)v_anchor})
        if (!aligned16(p)) return PCF_ERR_INVALID_ARG;
    if ((s = check_device()) != PCF_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(H[L_TOTAL_SEL] / kPage);
    const auto* kp = reinterpret_cast<const uint4*>(k_pool);
    const auto* vp = reinterpret_cast<const uint4*>(v_pool);
    auto* ka = reinterpret_cast<uint4*>(k_anchor);
    auto* va = reinterpret_cast<uint4*>(v_anchor);
    return H[L_D] == 128 ? launch(pack_anchor_kernel<128>, grid, dim3(256), 0, st, layout->dev, sel_idx, kp, vp, ka, va)
                         : launch(pack_anchor_kernel<64>, grid, dim3(256), 0, st, layout->dev, sel_idx, kp, vp, ka, va);
}

extern "C" pcf_status pcf_gather_rows(const pcf_layout* layout, const int32_t* sel_idx, const uint16_t* src,
                                      int32_t row_elems, uint16_t* dst, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (row_elems <= 0 || row_elems % 8 != 0) return PCF_ERR_INVALID_ARG;
    if (H[L_TOTAL_SEL] == 0) return PCF_OK;
    if (!sel_idx || !src || !dst || !aligned16(src) || !aligned16(dst)) return PCF_ERR_INVALID_ARG;
    if ((s = check_device()) != PCF_OK) return s;
    return launch(gather_kernel, dim3(H[L_TOTAL_SEL]), dim3(256), 0, static_cast<cudaStream_t>(stream), layout->dev,
                  sel_idx, reinterpret_cast<const uint4*>(src), row_elems / 8, reinterpret_cast<uint4*>(dst));
}

namespace {
pcf_status fused_attention_entry(const pcf_layout* layout, const uint16_t* q_fresh, const uint16_t* k_fresh,
                                 const uint16_t* v_fresh, const uint16_t* k_pool, const uint16_t* v_pool,
                                 const uint16_t* excl, const int32_t* row_pos, const float* rope, uint16_t* out,
                                 void* ws, size_t ws_bytes, cudaEvent_t ev_start, cudaEvent_t ev_stop, void* stream,
                                 bool paged) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (H[L_TOTAL_ROWS] == 0) {
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        if (ev_start && cudaEventRecord(ev_start, st) != cudaSuccess) return PCF_ERR_CUDA;
        if (ev_stop && cudaEventRecord(ev_stop, st) != cudaSuccess) return PCF_ERR_CUDA;
        return PCF_OK;
    }
    if (!q_fresh || !k_fresh || !v_fresh || !row_pos || !rope || !out || !ws) return PCF_ERR_INVALID_ARG;
    if (H[L_TOTAL_TOKENS] > 0 && (!k_pool || !v_pool || !excl)) return PCF_ERR_INVALID_ARG;
    const void* al[] = {q_fresh, k_fresh, v_fresh, rope, out, ws};
    for (const void* p : al)
        if (!aligned16(p)) return PCF_ERR_INVALID_ARG;
    if ((k_pool && !aligned16(k_pool)) || (v_pool && !aligned16(v_pool))) return PCF_ERR_INVALID_ARG;
    if (ws_bytes < (paged ? paged_ws(H).total : attn_ws(H).total)) return PCF_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_device()) != PCF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (paged)
        return H[L_D] == 128 ? paged_attention_impl<128>(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl,
                                                         row_pos, rope, out, ws, st, ev_start, ev_stop)
                             : paged_attention_impl<64>(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl,
                                                        row_pos, rope, out, ws, st, ev_start, ev_stop);
    return H[L_D] == 128 ? attention_impl<128>(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl, row_pos, rope,
                                               out, ws, st, ev_start, ev_stop)
                         : attention_impl<64>(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl, row_pos, rope,
                                              out, ws, st, ev_start, ev_stop);
}
}  // namespace

extern "C" pcf_status pcf_fused_attention(const pcf_layout* layout, const uint16_t* q_fresh, const uint16_t* k_fresh,
                                          const uint16_t* v_fresh, const uint16_t* k_pool, const uint16_t* v_pool,
                                          const uint16_t* excl, const int32_t* row_pos, const float* rope,
                                          uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
    return fused_attention_entry(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl, row_pos, rope, out, ws,
                                 ws_bytes, nullptr, nullptr, stream, false);
}

extern "C" pcf_status pcf_fused_attention_paged(const pcf_layout* layout, const uint16_t* q_fresh,
                                                const uint16_t* k_fresh, const uint16_t* v_fresh,
                                                const uint16_t* k_pool, const uint16_t* v_pool, const uint16_t* excl,
                                                const int32_t* row_pos, const float* rope, uint16_t* out, void* ws,
                                                size_t ws_bytes, void* stream) {
    return fused_attention_entry(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl, row_pos, rope, out, ws,
                                 ws_bytes, nullptr, nullptr, stream, true);
}

extern "C" pcf_status pcf_fused_attention_timed(const pcf_layout* layout, const uint16_t* q_fresh,
                                                const uint16_t* k_fresh, const uint16_t* v_fresh,
                                                const uint16_t* k_pool, const uint16_t* v_pool, const uint16_t* excl,
                                                const int32_t* row_pos, const float* rope, uint16_t* out, void* ws,
                                                size_t ws_bytes, void* ev_kernel_start, void* ev_kernel_stop,
                                                int32_t paged, void* stream) {
    if (!ev_kernel_start || !ev_kernel_stop) return PCF_ERR_INVALID_ARG;
    return fused_attention_entry(layout, q_fresh, k_fresh, v_fresh, k_pool, v_pool, excl, row_pos, rope, out, ws,
                                 ws_bytes, static_cast<cudaEvent_t>(ev_kernel_start),
                                 static_cast<cudaEvent_t>(ev_kernel_stop), stream, paged != 0);
}

extern "C" pcf_status pcf_copy_async(int32_t n, void* const* dst, const void* const* src, const size_t* bytes,
                                     void* stream) {
    if (n < 0 || (n > 0 && (!dst || !src || !bytes))) return PCF_ERR_INVALID_ARG;
    if (n == 0) return PCF_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PCF_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int32_t i = 0; i < n; ++i)
        if (bytes[i] > 0 && cudaMemcpyAsync(dst[i], src[i], bytes[i], cudaMemcpyDefault, st) != cudaSuccess)
            return PCF_ERR_CUDA;
    return PCF_OK;
}

extern "C" pcf_status pcf_prefetch_pool_pages(const pcf_layout* layout, const uint16_t* src_k, const uint16_t* src_v,
                                              uint16_t* dst_k, uint16_t* dst_v, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (!src_k || !dst_k || (!src_v) != (!dst_v)) return PCF_ERR_INVALID_ARG;
    // the physical page runs the layout's spans reference, each once; touching runs merge
    std::vector<std::pair<int64_t, int64_t>> runs;   // [first page, end page)
    const int32_t* SP = H + H[L_OFF_SPAN];
    for (int i = 0; i < H[L_N_SPANS]; ++i) {
        const int64_t a = SP[i * S_STRIDE + S_PHYS_FIRST], n = SP[i * S_STRIDE + S_N_PAGES];
        if (a < 0 || n < 0 || a + n > H[L_N_PHYS]) return PCF_ERR_INVALID_ARG;
        if (n > 0) runs.emplace_back(a, a + n);
    }
    std::sort(runs.begin(), runs.end());
    std::vector<std::pair<int64_t, int64_t>> merged;
    for (const auto& r : runs) {
        if (!merged.empty() && r.first <= merged.back().second) merged.back().second = std::max(merged.back().second, r.second);
        else merged.push_back(r);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PCF_ERR_NO_DEVICE;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t page_elems = (int64_t)H[L_HKV] * kPage * H[L_D];   // one page, every kv head
    for (const auto& r : merged) {
        const int64_t off = r.first * page_elems;
        const size_t bytes = (size_t)((r.second - r.first) * page_elems) * 2;
        if (cudaMemcpyAsync(dst_k + off, src_k + off, bytes, cudaMemcpyDefault, st) != cudaSuccess) return PCF_ERR_CUDA;
        if (src_v && cudaMemcpyAsync(dst_v + off, src_v + off, bytes, cudaMemcpyDefault, st) != cudaSuccess)
            return PCF_ERR_CUDA;
    }
    return PCF_OK;
}

extern "C" pcf_status pcf_wait_limit_check(int64_t limit_cycles, int32_t* flag, void* stream) {
    if (limit_cycles < 1000 || limit_cycles > 200000000LL || !flag || (reinterpret_cast<uintptr_t>(flag) & 3u))
        return PCF_ERR_INVALID_ARG;
    pcf_status s = check_device();
    if (s != PCF_OK) return s;
    return launch(wait_limit_check_kernel, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream),
                  (long long)limit_cycles, flag);
}

extern "C" pcf_status pcf_check_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PCF_ERR_CUDA;
    int code = 0;
    if (cudaMemcpyFromSymbol(&code, g_pcf_dev_error, sizeof(int)) != cudaSuccess) return PCF_ERR_CUDA;
    if (code != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_pcf_dev_error, &zero, sizeof(int)) != cudaSuccess) return PCF_ERR_CUDA;
    }
    if (code == kDevErrTimeout) return PCF_ERR_DEVICE_TIMEOUT;
    if (code == kDevErrBounds) return PCF_ERR_DEVICE_BOUNDS;
    if (code == kDevErrRange) return PCF_ERR_DEVICE_RANGE;
    return PCF_OK;
}

// ------------------------------------------------------------------ allocation-free scoring
// Scoring with its scratch inside the library image instead of a caller buffer, for callers that
// must not allocate device memory on this path (see pcf_score_noalloc in pcf.h).  Every GPU that
// loads the library holds this array until the process exits; all calls on a device share it.
static __device__ __align__(256) uint8_t g_pcf_noalloc_ws[PCF_SCORE_NOALLOC_MAX_WORKSPACE];

namespace {
std::mutex g_noalloc_mu;
// (device ordinal, CUDA context) -> device address of g_pcf_noalloc_ws.  Keyed on the context as
// well: if the device's primary context is torn down and created again (cudaDeviceReset), the
// module is loaded anew and the array may sit at another address.
std::map<std::pair<int, void*>, void*> g_noalloc_ptr;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;

// The array's name is only a host-side stand-in in host code; its device address is looked up
// once per device and context, with that device current.
pcf_status noalloc_workspace(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PCF_ERR_NO_DEVICE;
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
    });
    CUcontext ctx = nullptr;
    if (!g_ctx_get || g_ctx_get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PCF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const auto key = std::make_pair(dev, static_cast<void*>(ctx));
    auto it = g_noalloc_ptr.find(key);
    if (it == g_noalloc_ptr.end()) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pcf_noalloc_ws) != cudaSuccess || p == nullptr) return PCF_ERR_CUDA;
        it = g_noalloc_ptr.emplace(key, p).first;
    }
    *out = it->second;
    return PCF_OK;
}
}  // namespace

extern "C" pcf_status pcf_score_noalloc(const pcf_layout* layout, const uint16_t* q_query, const uint16_t* k_pool,
                                        const float* rope, float* importance, void* stream) {
    pcf_status s = check_layout(layout);
    if (s != PCF_OK) return s;
    const int32_t* H = layout->host;
    if (H[L_TOTAL_TOKENS] == 0) return PCF_OK;
    if (!k_pool || !rope || !importance || (H[L_TOTAL_QUERY] > 0 && !q_query)) return PCF_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(rope) || (q_query && !aligned16(q_query))) return PCF_ERR_INVALID_ARG;
    if (score_ws(H).total > PCF_SCORE_NOALLOC_MAX_WORKSPACE) return PCF_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_device()) != PCF_OK) return s;
    void* ws = nullptr;
    if ((s = noalloc_workspace(&ws)) != PCF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return H[L_D] == 128 ? score_impl<128>(layout, q_query, k_pool, rope, importance, ws, st)
                         : score_impl<64>(layout, q_query, k_pool, rope, importance, ws, st);
}
