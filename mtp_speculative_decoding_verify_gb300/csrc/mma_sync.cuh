// Warp-level bf16 tensor-core helpers (mma.sync m16n8k16, ldmatrix) and
// the 128-byte-swizzled shared-memory addressing that matches TMA tiles
// written with CU_TENSOR_MAP_SWIZZLE_128B (rows of 64 bf16 = 128 B; the
// 16-byte chunk c of row r sits at chunk c ^ (r % 8)).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace mtp {
namespace mma {

// Byte offset of element (row, col) in a [rows][64] bf16 box with 128-B
// swizzling; col must be a multiple of 8 (one 16-byte chunk).
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7))) << 4));
}

// Byte offset of (row, col) in a tile of `rows` rows stored as consecutive
// 64-column boxes (box b holds columns 64b .. 64b+63).
__device__ __forceinline__ uint32_t sw128_boxed(int rows, int row, int col) {
  return (uint32_t)((col >> 6) * rows * 128) + sw128(row, col & 63);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// C[16x8] += A[16x16] * B[16x8], bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace mma
}  // namespace mtp
