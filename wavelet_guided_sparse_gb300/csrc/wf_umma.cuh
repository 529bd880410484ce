// Fifth-generation tensor-core helpers (tcgen05, sm_100 family): tensor-
// memory allocation, shared-memory matrix descriptors, the single-thread
// bf16 MMA with an fp32 accumulator in tensor memory, its completion signal
// and the accumulator read-back.
//
// Operand layouts: the queries use the "core-matrix" K-major layout without
// swizzle; the A operands use its 128-byte-swizzled form (sw_offset below).
// Core-matrix layout:
// a matrix of R rows x K bf16 values is stored as 8-row x 16-byte core
// matrices; element (r, k) sits at byte
//     (r / 8) * sbo + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2,
// i.e. the core matrices of one 8-row group are contiguous along K
// (leading byte offset 128) and consecutive 8-row groups are sbo = K * 16
// bytes apart (stride byte offset).  Every 16-byte row chunk is contiguous,
// so ldmatrix can read the same layout (one chunk address per lane).
#pragma once

#include <stdint.h>

#include "wf_common.cuh"

namespace wf {

// Byte offset of row r, 16-byte chunk ch in the core-matrix layout.
__device__ __forceinline__ uint32_t cm_offset(int r, int ch, int sbo) {
  return static_cast<uint32_t>((r >> 3) * sbo + ch * 128 + (r & 7) * 16);
}

// 128-byte-swizzled K-major layout (the MMA A operands written row by row):
// K is cut into 64-element (128-byte) column blocks of m_alloc rows each,
// 128 bytes per row, 8-row groups 1024 bytes apart, and the 16-byte chunk c
// of row r sits at chunk position c ^ (r % 8) of its 128-byte line.  The
// eight chunks of a row half therefore fill one line: row-wise stores are
// free of bank conflicts.  The region must start on a 1024-byte boundary.
__device__ __forceinline__ uint32_t sw_offset(int r, int ch, int m_alloc) {
  return static_cast<uint32_t>((ch >> 3) * (m_alloc * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                               (((ch & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- tensor copies
// 2-D tiled tensor copy global -> shared (TMA engine) of the box at column x,
// row y of the tensor map (a __grid_constant__ kernel parameter), completion
// counted in bytes on `bar`.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Brings a tensor map (kernel parameter) into the descriptor cache ahead of
// its first tensor copy.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------- tensor memory
// Allocates ncols (power of two, 32..512) columns of tensor memory for this
// CTA; one whole warp executes it and the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Ordering of tcgen05 operations across a thread barrier.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor: K-major, no swizzle, base offset 0.
//   bits 0-13  start address >> 4     bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4  bits 46-47 descriptor version (1)
//   bits 61-63 swizzle mode (0: none)
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Descriptor of the 128-byte-swizzled K-major layout (swizzle mode 2,
// stride byte offset 1024, leading byte offset unused); a K step inside a
// 128-byte line advances the start address by 2 bytes per element.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32
// accumulator, M x N tile (M = 64 or 128; N a multiple of 8 (M = 64) or 16).
//   bits 4-5 accumulator format (1: f32)  bits 7-9 / 10-12 A / B format (1: bf16)
//   bit 15 / 16 A / B major (0: K)  bits 17-22 N >> 3  bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- MMA
// D[tmem] (+)= A * B^T over one K = 16 step; issued by a single thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- read-back
// Lane l of the calling warp receives columns [col, col + 16) of tensor-
// memory lane (warp % 4) * 32 + l; taddr carries that lane base and column.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Issue-only form of tmem_ld16 (no wait): several loads can be in flight
// before one tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace wf
