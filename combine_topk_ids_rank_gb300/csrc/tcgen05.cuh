// tcgen05.cuh -- inline-PTX wrappers for the sm_100-family tensor cores
// (tcgen05: MMA from shared-memory descriptors into tensor memory) and the
// tiled TMA load, as used by expert_gemm.cu.
//
// Encodings (PTX ISA, "Tensor Memory" and "tcgen05.mma" sections):
//  * shared-memory matrix descriptor (64 bits): start address >> 4 in
//    [0,14), leading-dimension byte offset >> 4 in [16,30), stride-dimension
//    byte offset >> 4 in [32,46), the constant 0b001 in [46,49), base offset
//    in [49,52), swizzle mode in [61,64) (2 = 128-byte swizzle);
//  * instruction descriptor of .kind::f16 / .kind::f8f6f4 (32 bits): D
//    format in [4,6) (1 = f32), A format in [7,10) and B format in [10,13)
//    (f16 kind: 1 = bf16; f8f6f4 kind: 0 = E4M3),
//    A / B major in bits 15 / 16 (0 = K-major), N >> 3 in [17,23),
//    M >> 4 in [24,29);
//  * tensor-memory address: lane in bits [16,32), column in [0,16).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moe {
namespace tc {

// K-major operand tile staged by a 128-byte-swizzled TMA load: rows of
// 128 bytes (64 bf16), 8-row groups 1024 bytes apart.  The tile must start
// on a 1024-byte boundary.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)(16u >> 4) << 16;                // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;                          // fixed 0b001
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// bf16 x bf16 -> f32, both operands K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// e4m3 x e4m3 -> f32 (.kind::f8f6f4, format code 0 = E4M3), both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Allocation of `ncols` tensor-memory columns (a power of two >= 32) by one
// whole warp; the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     ptx::smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T on 8-bit operands (32 per K step).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The mbarrier receives one arrival when every tcgen05 operation issued so
// far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            ptx::smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 columns of 32-bit accumulators: thread i of the warp gets
// lane (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void ld_32x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 2-D tiled TMA load of the box at (x = inner coordinate, y) into shared
// memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(ptx::smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(ptx::smem_u32(bar))
        : "memory");
}

}  // namespace tc
}  // namespace moe
