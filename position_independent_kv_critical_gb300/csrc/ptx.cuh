// Thin inline-PTX wrappers for sm_103a: mbarriers with bounded waits, TMA (cp.async.bulk),
// tcgen05 (TMEM alloc / MMA / commit / ld / st) and UMMA shared-memory descriptors.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pcf {

enum : int { kDevErrNone = 0, kDevErrTimeout = 1, kDevErrBounds = 2, kDevErrRange = 3 };

// Device error word of this library (one per loaded module); read and cleared by
// pcf_check_device_error.  Defined here: the library is a single CUDA translation unit.
__device__ int g_pcf_dev_error = 0;

__device__ __forceinline__ void set_dev_error(int code) { atomicCAS(&g_pcf_dev_error, 0, code); }

// About 1 s at GB300 clocks: no correct pipeline wait comes anywhere near this.
constexpr long long kWaitLimitCycles = 2000000000LL;

// ---------------------------------------------------------------- programmatic dependent launch
// The library's kernels are launched with programmatic stream serialization, so a kernel's CTAs
// may start while the previous kernel in the stream is still running.  Everything before
// grid_dep_wait() may touch only data no kernel writes (the layout, tensor maps, shared memory);
// grid_dep_wait() returns once the previous grid has finished and its writes are visible (and,
// since every kernel here waits before it finishes, every earlier grid too).  grid_dep_launch()
// lets the next grid start its own prologue.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok;
}

// the same with a suspend-time hint: a waiting thread sleeps up to `ns` nanoseconds (or until the
// phase completes) instead of polling, which keeps idle warps off the shared-memory pipe
__device__ __forceinline__ uint32_t mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok;
}
// non-blocking test of the same
__device__ __forceinline__ uint32_t mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok;
}

// Bounded wait for the phase of `parity` to complete.  Returns false (and raises the CTA's abort
// flag plus the device error word) when `limit` cycles run out or another role already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          long long limit = kWaitLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            set_dev_error(kDevErrTimeout);
            return false;
        }
    }
}

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles / 4) {
            set_dev_error(kDevErrTimeout);
            return;
        }
    }
}

// ---------------------------------------------------------------- cross-CTA hand-off
// "Last one finishes the job": a CTA's threads write their results, meet at a CTA barrier, and one
// thread adds 1 to a counter with acquire-release semantics at GPU scope.  The release makes
// everything the CTA wrote before the barrier visible with the increment (release is cumulative);
// the acquire lets the CTA that sees the final count read what every other CTA wrote, once its
// other threads are ordered after that thread by a second CTA barrier.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---------------------------------------------------------------- proxies / fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA / bulk copies
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// L2 prefetch of one tile of a 2D tensor map (no shared memory, no barrier)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, one CTA.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Four K = 16 steps of D[tmem] (+)= A[smem] * B[smem]^T in one block, for a warp that runs the
// issue loop converged: every lane executes it, only `leader`'s predicate issues.  The operands
// are 128-byte-swizzled K-major: step kk starts 32 bytes further along K, i.e. 2 more in the low
// word of both descriptors (whose high words, `hi`, stay fixed).  Building the descriptors in the
// block keeps their arithmetic next to the instructions that use them.
__device__ __forceinline__ void mma_ss_k4(uint32_t leader, uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                          uint32_t hi, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred L, p, t;\n\t.reg .b64 da, db;\n\t.reg .b32 la, lb;\n\t"
        "setp.ne.b32 L, %0, 0;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.eq.b32 t, %0, %0;\n\t"
        "mov.b64 da, {%2, %4};\n\tmov.b64 db, {%3, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, p;\n\t"
        "add.u32 la, %2, 2;\n\tadd.u32 lb, %3, 2;\n\t"
        "mov.b64 da, {la, %4};\n\tmov.b64 db, {lb, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
        "add.u32 la, %2, 4;\n\tadd.u32 lb, %3, 4;\n\t"
        "mov.b64 da, {la, %4};\n\tmov.b64 db, {lb, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
        "add.u32 la, %2, 6;\n\tadd.u32 lb, %3, 6;\n\t"
        "mov.b64 da, {la, %4};\n\tmov.b64 db, {lb, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t}\n" ::"r"(leader),
        "r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Four K = 16 steps of D[tmem] (+)= A[tmem] * B[smem]^T (A: 8 TMEM columns a step; B MN-major,
// 128-byte swizzle, 2048 bytes a step, i.e. 128 more in the descriptor's low word).
__device__ __forceinline__ void mma_ts_k4(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                          uint32_t hi, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred L, p, t;\n\t.reg .b64 db;\n\t.reg .b32 ta, lb;\n\t"
        "setp.ne.b32 L, %0, 0;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.eq.b32 t, %0, %0;\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], db, %5, p;\n\t"
        "add.u32 ta, %2, 8;\n\tadd.u32 lb, %3, 128;\n\tmov.b64 db, {lb, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, t;\n\t"
        "add.u32 ta, %2, 16;\n\tadd.u32 lb, %3, 256;\n\tmov.b64 db, {lb, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, t;\n\t"
        "add.u32 ta, %2, 24;\n\tadd.u32 lb, %3, 384;\n\tmov.b64 db, {lb, %4};\n\t"
        "@L tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, t;\n\t}\n" ::"r"(leader),
        "r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
// tcgen05.commit by `leader` only (the lane that issued the MMAs), the warp converged.
__device__ __forceinline__ void mma_commit_by(uint32_t leader, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred L;\n\tsetp.ne.b32 L, %0, 0;\n\t"
        "@L tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}\n" ::"r"(leader),
        "r"(smem_u32(bar))
        : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

#define PCF_R32(a) "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), \
    "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),          \
    "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),        \
    "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31])
#define PCF_W32(a) "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), \
    "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15]),          \
    "r"(a[16]), "r"(a[17]), "r"(a[18]), "r"(a[19]), "r"(a[20]), "r"(a[21]), "r"(a[22]), "r"(a[23]),        \
    "r"(a[24]), "r"(a[25]), "r"(a[26]), "r"(a[27]), "r"(a[28]), "r"(a[29]), "r"(a[30]), "r"(a[31])

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32*(w%4)..+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : PCF_R32(r)
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        PCF_W32(r)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// UMMA shared-memory descriptor, 128-byte swizzle, K-major: rows of 128 bytes, 8-row groups
// 1024 bytes apart (stride byte offset); the leading byte offset is unused for this layout.
// Bits: [0,14) start>>4, [16,30) LBO>>4, [32,46) SBO>>4, [46,48) version 1, [61,64) swizzle=2.
__device__ __forceinline__ uint64_t desc_sw128_kmajor(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// 128-byte-swizzle descriptors as two 32-bit words (K-major as above with lbo 16; MN-major with
// lbo = the byte distance between 64-wide atoms along N): the low word holds the start address
// and the leading byte offset, the high word (fixed) the 1024-byte stride, version and swizzle.
__device__ __forceinline__ uint32_t desc_sw128_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr & 0x3FFFFu) >> 4) | ((lbo_bytes >> 4) << 16);
}
constexpr uint32_t kDescSw128Hi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));
// Offset, in descriptor units (16 bytes, added to the start-address field), of K = 16 step kk of a
// 128-byte-swizzled K-major operand whose rows hold 64 elements of K per 1024-byte-stride atom
// column (atoms of 64 K elements are `atom_bytes` apart): 32 bytes a step inside an atom.  The
// start field cannot carry into the next field: shared addresses stay below 2^18 bytes.
__host__ __device__ constexpr uint64_t sw128_k_step(int kk, uint32_t atom_bytes = 16384) {
    return (uint64_t)(((uint32_t)(kk >> 2) * atom_bytes + (uint32_t)(kk & 3) * 32u) >> 4);
}
// UMMA shared-memory descriptor, no swizzle, K-major: 8-row x 16-byte core matrices; `k_stride`
// bytes between core matrices adjacent along K, `row_stride` bytes between 8-row groups.
__device__ __forceinline__ uint64_t desc_noswz_kmajor(uint32_t saddr, uint32_t k_stride, uint32_t row_stride) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(k_stride >> 4) << 16) |
           ((uint64_t)(row_stride >> 4) << 32) | ((uint64_t)1 << 46);
}
// Byte offset of element (row, k) of a [rows][16] 16-bit slab in that layout (k_stride 128,
// row_stride 256).
__device__ __forceinline__ uint32_t slab16_off(uint32_t row, uint32_t k) {
    return (row >> 3) * 256u + (k >> 3) * 128u + (row & 7u) * 16u + (k & 7u) * 2u;
}
// Instruction descriptor, kind::f16: D fp32, A = B = bf16, A K-major, B K- or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Same with A = B = fp16 (format code 0): used for the rotated Q / K contractions.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// packed fp32 pairs (sm_100 and later issue one instruction for both halves)
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// a * b + c on both halves
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// the two bf16 halves of a 32-bit word as a packed fp32 pair (exact)
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v) {
    return f2_pack(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Rotated queries and keys are held in fp16 (10-bit mantissa, same tensor-core rate as bf16):
// saturating conversion, |values| above 65504 clamp to the largest finite fp16.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Largest magnitude that rounds to a finite fp16 (65504 plus half a unit in the last place).
constexpr float kF16Limit = 65520.0f;
// The same, recording in `big` (as the running maximum of |lo|, |hi|) whether a value was out of
// fp16 range; the caller raises kDevErrRange once for the whole row instead of clamping silently.
__device__ __forceinline__ uint32_t pack_f16x2_track(float lo, float hi, float& big) {
    big = max3f(big, fabsf(lo), fabsf(hi));
    return pack_f16x2(lo, hi);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a 128-byte-swizzled block
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace pcf
