// Thin wrappers over the sm_100-family tensor-core PTX (tcgen05) used by the
// prefill grouped GEMMs: tensor-memory allocation, the MMA from shared-memory
// operand descriptors, commit to an mbarrier, and tensor-memory loads.
#pragma once

#include <stdint.h>

#include "async_copy.cuh"

namespace moeq4k {
namespace tc {

// Byte offset of element (row r, k) inside a K-major tile of 64 fp16 per row
// stored with the 128-byte swizzle: 8-row groups of 1024 B, 128 B per row,
// 16-byte chunk j of row r stored at chunk position j ^ (r % 8).
__host__ __device__ inline uint32_t sw128_offset(int r, int k) {
    return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) +
                    (k & 7) * 2);
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// whose 8-row groups are 1024 B apart; `saddr` must lie in a 1024-byte
// aligned tile (plus the 32-byte K offset of the 16-wide slice).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFF);  // start address / 16
    d |= uint64_t(1) << 16;                // leading byte offset (unused in this layout)
    d |= uint64_t(1024 >> 4) << 32;        // stride byte offset: next 8-row group
    d |= uint64_t(1) << 46;                // descriptor version of the sm_100 family
    d |= uint64_t(2) << 61;                // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 D, both
// operands K-major, M x N.
__host__ __device__ inline uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Instruction descriptor of kind::tf32 (A and B tf32, type code 2), fp32 D,
// both operands K-major, M x N.
__host__ __device__ inline uint32_t idesc_tf32_f32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with tf32 operands (the fp32 values in
// shared memory, of which the MMA uses the tf32 part), issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void commit_arrive(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Each thread of the warp reads 8 consecutive fp32 columns of its TMEM lane.
// The destination registers hold the data only after tcgen05.wait::ld, so
// the wait takes them as read-write operands: no use of them can be
// scheduled between the load and the wait.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}

// 32-byte global store of eight fp32 values (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float *p, const float (&v)[8]) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]),
                 "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

// 16-byte cp.async that writes zeros when `valid` is false (no global read).
__device__ __forceinline__ void cp_async_16_zfill(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

}  // namespace tc
}  // namespace moeq4k
