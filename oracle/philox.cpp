/* Oracle: counter-based random numbers for the acceptance step
 * (test infrastructure only; see oracle.h).
 *
 * Philox4x32-10 as defined by Salmon, Moraes, Dror and Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3" (SC'11), section 3.2: each round multiplies
 * words 0 and 2 by the two Philox multipliers, swaps the halves and mixes in
 * the key; the key is bumped by the two Weyl constants between rounds.
 *
 * Stream layout (the pages do not fix one; this is the library's contract):
 *   key     = (seed low 32 bits, seed high 32 bits)
 *   counter = (request b, row j, vocab index v, tag)
 *   tag 1   accept uniform of row j: word 0 of counter (b, j, 0, 1)
 *   tag 2   race exponential, residual sample at the first rejection
 *   tag 3   race exponential, bonus sample when every draft is accepted
 * The race variate of vocabulary index v takes output word v mod 4 of
 * counter (b, j, floor(v / 4), tag): each generator call yields four
 * independent words, one per consecutive vocabulary entry.
 */
#include <math.h>
#include "oracle.h"

static const uint32_t kPhiloxM0 = 0xD2511F53u;
static const uint32_t kPhiloxM1 = 0xCD9E8D57u;
static const uint32_t kWeyl0 = 0x9E3779B9u;
static const uint32_t kWeyl1 = 0xBB67AE85u;

extern "C" void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += kWeyl0;
      k1 += kWeyl1;
    }
    uint64_t prod0 = (uint64_t)kPhiloxM0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)kPhiloxM1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static uint32_t philox_word0(uint64_t seed, uint32_t b, uint32_t j, uint32_t v, uint32_t tag) {
  uint32_t ctr[4] = {b, j, v, tag};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return out[0];
}

/* U in [0, 1) on a 2^-24 grid: the top 24 bits of word 0. */
extern "C" float oracle_accept_uniform(uint64_t seed, uint32_t b, uint32_t j) {
  uint32_t x = philox_word0(seed, b, j, 0u, 1u);
  return (float)(x >> 8) * 0x1p-24f;
}

/* E = -ln(1 - u), u = x * 2^-32 (x converted to binary32 with round to
 * nearest), evaluated as -log1p(-u) in binary32: an Exp(1) variate whose
 * resolution near 0 (the race winners) is 2^-32. */
extern "C" float oracle_race_exponential(uint64_t seed, uint32_t b, uint32_t j, uint32_t v, uint32_t tag) {
  uint32_t ctr[4] = {b, j, v / 4u, tag};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  uint32_t x = out[v % 4u];
  float u = (float)x * 0x1p-32f;
  return -log1pf(-u);
}
