// gs_ptx.cuh -- inline-PTX helpers for sm_103a: mbarriers, bulk async copies
// (TMA, global -> shared), proxy fences, and the bounded wait every kernel
// uses so that a copy that never lands ends the kernel with an error word
// instead of a hang.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gs {

// Device error word bits (see gs_device_status in include/gs.h).
constexpr unsigned kDevErrTimeout = 1u;    // a bounded wait gave up

// A wait gives up after this long (ns of %globaltimer); copies land in
// microseconds, so only a broken pipeline ever reaches it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (the copy engine).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses before later async-proxy
// (bulk copy) accesses to shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with `parity` to complete; gives up after `limit_ns`
// (default kWaitLimitNs), records kDevErrTimeout in *err and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, unsigned *err,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            if (err) atomicOr(err, kDevErrTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bulk asynchronous copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to this CTA's shared memory; completion is counted in
// bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (cp.async, cached in L2 only);
// src_bytes < 16 zero-fills the rest, 0 writes sixteen zero bytes without
// reading `src`.  Completion is tracked per thread in commit groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// 4-byte asynchronous copy global -> shared (cp.async through L1); src_bytes 0
// writes a zero word without reading `src`.  For element-wise transposing
// copies that 16-byte runs cannot do.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Waits until at most `pending` (0, 1 or 2; more counts as 2) of this thread's
// most recent commit groups are still in flight.
__device__ __forceinline__ void cp_async_wait_pending(int pending) {
    if (pending <= 0) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else if (pending == 1) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
        asm volatile("cp.async.wait_group 2;" ::: "memory");
    }
}

// Packed fp32 pairs (Blackwell FMUL2 / FFMA2 through the CUDA builtins, so the
// compiler allocates the register pairs itself): lane-wise a*b and a*b+c, each
// rounded to nearest exactly as fmulf / fmaf would round it.
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
    return __ffma2_rn(a, b, c);
}

}  // namespace gs

// ------------------------------------------------------------------ tcgen05
//
// Fifth-generation tensor-core MMA with the accumulator in tensor memory
// (TMEM).  Operands are read from shared memory through 64-bit matrix
// descriptors; one thread issues the MMAs, completion is signalled on an
// mbarrier by tcgen05.commit, and the accumulator is read back with
// tcgen05.ld.

namespace gs {

// Shared-memory matrix descriptor, K-major operand without swizzling: the
// tile is made of 8-row x 16-byte core matrices (each 128 contiguous bytes);
// `lbo` is the byte distance between core matrices adjacent along K, `sbo`
// between core matrices adjacent along M (or N).
__device__ __forceinline__ uint64_t umma_desc_kmajor(uint32_t smem_addr, uint32_t lbo,
                                                     uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;          // leading-dimension byte offset
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;          // stride-dimension byte offset
    d |= (uint64_t)1 << 46;                               // descriptor version for tcgen05
    // base offset 0, relative leading-dimension offsets, no swizzling (bits 61-63 = 0)
    return d;
}

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle:
// each row (M or N index) holds 64 two-byte K elements in 128 bytes, 8 rows
// form a 1024-byte atom, and the 16-byte chunk c of row r is stored at chunk
// c ^ (r % 8) of that row (the atom must be 1024-byte aligned).  `sbo` is the
// byte distance between 8-row atoms; a K step of 16 elements inside the atom
// moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t umma_desc_kmajor_sw128(uint32_t smem_addr, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1 << 16;                               // leading offset: unused with this swizzle
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;          // stride-dimension byte offset
    d |= (uint64_t)1 << 46;                               // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                               // 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, A and B both bf16
// (is_bf16) or both fp16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(bool is_bf16, int M, int N) {
    return (1u << 4)                                    // D format: fp32
           | ((is_bf16 ? 1u : 0u) << 7)                 // A format
           | ((is_bf16 ? 1u : 0u) << 10)                // B format
           | ((uint32_t)(N >> 3) << 17)                 // N / 8
           | ((uint32_t)(M >> 4) << 24);                // M / 16
}

// Allocate `ncols` TMEM columns (a power of two >= 32); the whole warp calls
// it; the TMEM address lands in shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T for one M x N x 16 step.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tcgen05_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tcgen05_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// Eight consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace gs
