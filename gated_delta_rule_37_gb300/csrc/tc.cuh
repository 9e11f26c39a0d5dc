// Blackwell (sm_103a) building blocks written as inline PTX: shared-memory
// matrix descriptors and swizzled tile addressing for tcgen05.mma, tensor
// memory allocation and loads, mbarriers with bounded waits, 1-D bulk copies.
//
// Layout conventions (bf16 operands, byte offsets inside a 1024-aligned tile):
//   K-major, 128-byte swizzle ("k128"): the contraction index runs along a
//     128-byte row; an operand with rows r and contraction index k is stored
//     in column blocks of 64 elements, each block [rows][64] with rows of 128
//     bytes, 8-row atoms of 1024 bytes, 16-byte chunk c of row r stored at
//     chunk c ^ (r % 8).  Descriptor: SBO = 1024, layout SWIZZLE_128B.
//   MN-major, 128-byte swizzle: the non-contraction index runs along the row.
//     A tile [k rows][n] with n split in atoms of 64 elements is byte-identical
//     to the K-major tile of the same [rows][cols] array, so one staged tile
//     serves as a K-major operand (contracting over its columns) and as an
//     MN-major operand (contracting over its rows).  Descriptor: LBO = stride
//     between 64-element atoms (rows * 128), SBO = 1024.
//   MN-major, 64-byte swizzle ("mn64"): for 32-element wide operands; row k
//     of 64 bytes, 8-row groups of 512 bytes, chunk c ^ ((k % 8) / 2).
//     Descriptor: LBO = SBO = 512, layout SWIZZLE_64B.
// Accumulators (fp32, cta_group::1): M = 128 puts row r in TMEM lane r; M = 64
// puts row r in lane 32 * (r / 16) + r % 16.  Warp w reads lanes
// 32 * (w % 4) .. + 31.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdr {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- swizzled tile offsets (bytes) ------------------------------------------
__device__ __forceinline__ uint32_t off_k128(int row, int col, int rows) {
    const int cb = col >> 6, kk = col & 63;
    return cb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((((kk >> 3) ^ (row & 7))) << 4) + (kk & 7) * 2;
}
// byte offset of the 16-byte chunk holding columns [8*ch, 8*ch+8) of `row`
__device__ __forceinline__ uint32_t chunk_k128(int row, int ch, int rows) {
    const int cb = ch >> 3, c = ch & 7;
    return cb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
}
// MN-major 64-byte swizzle, 32-element rows: chunk ch (0..3) of row k
__device__ __forceinline__ uint32_t chunk_mn64(int k, int ch) {
    return (k >> 3) * 512 + (k & 7) * 64 + ((ch ^ ((k & 7) >> 1)) << 4);
}

// ---- descriptors ------------------------------------------------------------
enum : uint32_t { kSwizzleNone = 0, kSwizzle128 = 2, kSwizzle64 = 4, kSwizzle32 = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

// kind::f16 instruction descriptor: bf16 x bf16 -> fp32, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// n_steps (4 or 8) k-steps into one accumulator: descriptors advance by
// a_step[ks] / b_step per k-step (16-byte units); the first step overwrites D
// when `first`, every later one accumulates.
template <int kSteps>
__device__ __forceinline__ void mma_ksteps(uint32_t d_tmem, uint64_t a, const uint32_t (&a_step)[kSteps], uint64_t b,
                                           uint32_t b_step, uint32_t idesc, bool first) {
#pragma unroll
    for (int ks = 0; ks < kSteps; ++ks)
        mma_bf16(d_tmem, a + a_step[ks], b + (uint64_t)b_step * ks, idesc, (first && ks == 0) ? 0u : 1u);
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(mbar) : "memory");
}

// ---- tensor memory -----------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(slot_smem), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 64 consecutive fp32 columns (two 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
    uint32_t r[64];
#define GDR_LD32(base, off)                                                                                       \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                       \
                 : "=r"(r[base + 0]), "=r"(r[base + 1]), "=r"(r[base + 2]), "=r"(r[base + 3]), "=r"(r[base + 4]),  \
                   "=r"(r[base + 5]), "=r"(r[base + 6]), "=r"(r[base + 7]), "=r"(r[base + 8]), "=r"(r[base + 9]),  \
                   "=r"(r[base + 10]), "=r"(r[base + 11]), "=r"(r[base + 12]), "=r"(r[base + 13]),                 \
                   "=r"(r[base + 14]), "=r"(r[base + 15]), "=r"(r[base + 16]), "=r"(r[base + 17]),                 \
                   "=r"(r[base + 18]), "=r"(r[base + 19]), "=r"(r[base + 20]), "=r"(r[base + 21]),                 \
                   "=r"(r[base + 22]), "=r"(r[base + 23]), "=r"(r[base + 24]), "=r"(r[base + 25]),                 \
                   "=r"(r[base + 26]), "=r"(r[base + 27]), "=r"(r[base + 28]), "=r"(r[base + 29]),                 \
                   "=r"(r[base + 30]), "=r"(r[base + 31])                                                           \
                 : "r"(taddr + (off)))
    GDR_LD32(0, 0);
    GDR_LD32(32, 32);
#undef GDR_LD32
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
}

// ---- mbarriers ----------------------------------------------------------------
// Bounded waits: a wait gives up after kWaitLimitNs of wall time (read from
// %globaltimer) and reports failure so the kernel can record an error and
// leave instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(mbar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" :: "r"(mbar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred P1;\n\tmbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
                 "selp.b32 %0, 1, 0, P1;\n\t}\n" : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_test(uint32_t mbar, uint32_t parity);

// Returns false if the wait gave up or `abort` (shared flag) was raised.  A
// phase that has already completed is detected with a non-suspending test.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, volatile int* abort) {
    if (mbar_test(mbar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(mbar, parity)) return true;
        if ((i & 255) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// Wait for bulk copies to land regardless of any abort: copies complete on
// their own, and none may still be writing shared memory when the CTA exits.
__device__ __forceinline__ bool mbar_wait_copies(uint32_t mbar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try(mbar, parity)) return true;
        if ((i & 255) == 255 && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---- 1-D bulk copy global -> shared, completing on an mbarrier --------------
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst_smem), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}

// ---- 1-D bulk copy shared -> global (bulk-group completion) ---------------------
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" :: "l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of every committed bulk copy have been read
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk copy but the most recent group has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every committed bulk copy has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// L2 prefetch of `bytes` (multiple of 16) at a 16-byte aligned global address.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}
// L2 prefetch of the 16-byte aligned interior of [src, src + bytes).
__device__ __forceinline__ void prefetch_l2_span(const void* src, size_t bytes) {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(src) + 15) & ~uintptr_t(15);
    const uintptr_t b = (reinterpret_cast<uintptr_t>(src) + bytes) & ~uintptr_t(15);
    if (b > a) prefetch_l2(reinterpret_cast<const void*>(a), (uint32_t)(b - a));
}

// ---- programmatic dependent launch ---------------------------------------------
// Block until the grids this one depends on have completed and their writes are
// visible (a no-op for a normally launched kernel).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream, if launched as a dependent, to start.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- named barriers -------------------------------------------------------------
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Non-suspending variant for a single polling thread (the MMA issuers).
__device__ __forceinline__ bool mbar_test(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred P1;\n\tmbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
                 "selp.b32 %0, 1, 0, P1;\n\t}\n" : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_spin(uint32_t mbar, uint32_t parity, volatile int* abort) {
    if (mbar_test(mbar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(mbar, parity)) return true;
        if ((i & 255) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// 16 consecutive fp32 columns of this thread's lane from each of three
// addresses, one wait.
__device__ __forceinline__ void tmem_ld16x3(uint32_t a0, uint32_t a1, uint32_t a2, float* v) {
    uint32_t r[48];
#define GDR_LD16(base, addr)                                                                                \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
                 : "=r"(r[base + 0]), "=r"(r[base + 1]), "=r"(r[base + 2]), "=r"(r[base + 3]), "=r"(r[base + 4]), \
                   "=r"(r[base + 5]), "=r"(r[base + 6]), "=r"(r[base + 7]), "=r"(r[base + 8]), "=r"(r[base + 9]), \
                   "=r"(r[base + 10]), "=r"(r[base + 11]), "=r"(r[base + 12]), "=r"(r[base + 13]),              \
                   "=r"(r[base + 14]), "=r"(r[base + 15])                                                       \
                 : "r"(addr))
    GDR_LD16(0, a0);
    GDR_LD16(16, a1);
    GDR_LD16(32, a2);
#undef GDR_LD16
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 48; ++j) v[j] = __uint_as_float(r[j]);
}

// 16 consecutive fp32 columns of this thread's lane from each of two
// addresses, one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t a0, uint32_t a1, float* v) {
    uint32_t r[32];
#define GDR_LD16(base, addr)                                                                                \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
                 : "=r"(r[base + 0]), "=r"(r[base + 1]), "=r"(r[base + 2]), "=r"(r[base + 3]), "=r"(r[base + 4]), \
                   "=r"(r[base + 5]), "=r"(r[base + 6]), "=r"(r[base + 7]), "=r"(r[base + 8]), "=r"(r[base + 9]), \
                   "=r"(r[base + 10]), "=r"(r[base + 11]), "=r"(r[base + 12]), "=r"(r[base + 13]),              \
                   "=r"(r[base + 14]), "=r"(r[base + 15])                                                       \
                 : "r"(addr))
    GDR_LD16(0, a0);
    GDR_LD16(16, a1);
#undef GDR_LD16
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ---- bf16 packing -------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}
// Two values x0, x1 -> packed bf16 pairs hi = (bf16(x0), bf16(x1)) and
// lo = (bf16(x0 - hi0), bf16(x1 - hi1)).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(x0, x1);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16(x0 - h0, x1 - h1);
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}

}  // namespace tc
}  // namespace gdr
