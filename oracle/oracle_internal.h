/* Oracle-internal helpers (test infrastructure only; see oracle.h). */
#ifndef MTP_ORACLE_INTERNAL_H
#define MTP_ORACLE_INTERNAL_H

#include <stdint.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static inline float oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays NaN. */
static inline uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* Element i of a tensor of the given dtype, widened to double. */
static inline double oracle_load(const void* base, int dtype, int64_t i) {
  if (dtype == 0) return (double)((const float*)base)[i];
  return (double)oracle_bf16_to_f32(((const uint16_t*)base)[i]);
}

/* Store a double as the given dtype (double -> binary32 -> bf16). */
static inline void oracle_store(void* base, int dtype, int64_t i, double x) {
  float f = (float)x;
  if (dtype == 0) ((float*)base)[i] = f;
  else ((uint16_t*)base)[i] = oracle_f32_to_bf16(f);
}

/* Copy one element between tensors of the same dtype. */
static inline void oracle_copy_elem(void* dst, int64_t di, const void* src, int64_t si, int dtype) {
  if (dtype == 0) ((float*)dst)[di] = ((const float*)src)[si];
  else ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
}

#endif
