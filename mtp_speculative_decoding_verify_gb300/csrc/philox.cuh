// Philox4x32-10 counter-based generator on the device.
//
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): ten rounds of (two 32x32->64 multiplies, half swap, key xor); the
// key is advanced by the two Weyl constants before every round after the
// first. Stream contract of this library: key = (seed low, seed high);
// the accept uniform of row j takes word 0 of counter (request, j, 0, 1); the
// race variate of vocabulary index v takes word v % 4 of counter
// (request, row, v / 4, tag), so one generator call serves four consecutive
// vocabulary entries.
#pragma once

#include <stdint.h>

namespace mtp {

enum : uint32_t { kTagAccept = 1u, kTagResidual = 2u, kTagBonus = 3u };

// All four output words of counter (c0, c1, c2, c3).
__device__ __forceinline__ uint4 philox4(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  uint32_t k0 = static_cast<uint32_t>(seed);
  uint32_t k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo_a = 0xD2511F53u * c0;
    const uint32_t hi_a = __umulhi(0xD2511F53u, c0);
    const uint32_t lo_b = 0xCD9E8D57u * c2;
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi_b ^ c1 ^ k0;
    const uint32_t n2 = hi_a ^ c3 ^ k1;
    c0 = n0;
    c1 = lo_b;
    c2 = n2;
    c3 = lo_a;
  }
  return make_uint4(c0, c1, c2, c3);
}

__device__ __forceinline__ uint32_t philox_word0(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return philox4(seed, c0, c1, c2, c3).x;
}

// Accept uniform of row j: top 24 bits of word 0, U in [0, 1).
__device__ __forceinline__ float accept_uniform(uint64_t seed, uint32_t b, uint32_t j) {
  const uint32_t x = philox_word0(seed, b, j, 0u, kTagAccept);
  return __uint2float_rn(x >> 8) * 0x1p-24f;
}

// Exp(1) variate of a race word x: E = -log1p(-u), u = x * 2^-32 (x rounded
// to binary32), so winners (small E) keep 2^-32 resolution.
__device__ __forceinline__ float race_variate(uint32_t x) {
  const float u = __fmul_rn(__uint2float_rn(x), 0x1p-32f);
  return -log1pf(-u);
}

// Race word of vocabulary index v: word v % 4 of counter (b, j, v / 4, tag).
__device__ __forceinline__ uint32_t race_word(uint64_t seed, uint32_t b, uint32_t j, uint32_t v, uint32_t tag) {
  const uint4 w = philox4(seed, b, j, v >> 2, tag);
  const uint32_t k = v & 3u;
  return k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w;
}

__device__ __forceinline__ float race_exponential(uint64_t seed, uint32_t b, uint32_t j, uint32_t v, uint32_t tag) {
  return race_variate(race_word(seed, b, j, v, tag));
}

}  // namespace mtp
