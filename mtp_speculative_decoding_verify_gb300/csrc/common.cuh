// Shared device helpers of the GB300 verify-step library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtp_verify.h"

namespace mtp {

constexpr int kWarp = 32;
constexpr int kBlock = MTP_BLOCK_SIZE;
constexpr int kMaxRows = MTP_MAX_DRAFTS + 1;
constexpr float kTieRel = 1e-5f;

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

template <typename T> struct Num;
template <> struct Num<float> {
  __device__ __forceinline__ static float to_f(float x) { return x; }
  __device__ __forceinline__ static float from_f(float x) { return x; }
};
template <> struct Num<__nv_bfloat16> {
  __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Running softmax statistics of one row: max m, sum of exp(x - m), and the
// argmax (largest value, lowest index among equal values).
struct RowStat {
  float m;
  float s;
  float best;
  int idx;
};

__device__ __forceinline__ RowStat rowstat_empty() { return RowStat{-INFINITY, 0.0f, -INFINITY, 0x7fffffff}; }

// Merge two partial statistics (associative and commutative up to rounding
// of s; the argmax part is exact).
__device__ __forceinline__ RowStat rowstat_merge(RowStat a, RowStat b) {
  RowStat r;
  r.m = fmaxf(a.m, b.m);
  float sa = (a.s == 0.0f) ? 0.0f : a.s * expf(a.m - r.m);
  float sb = (b.s == 0.0f) ? 0.0f : b.s * expf(b.m - r.m);
  r.s = sa + sb;
  bool take_b = (b.best > a.best) || (b.best == a.best && b.idx < a.idx);
  r.best = take_b ? b.best : a.best;
  r.idx = take_b ? b.idx : a.idx;
  return r;
}

__device__ __forceinline__ RowStat warp_merge(RowStat v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    RowStat w;
    w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
    w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    w.best = __shfl_xor_sync(0xffffffffu, v.best, o);
    w.idx = __shfl_xor_sync(0xffffffffu, v.idx, o);
    v = rowstat_merge(v, w);
  }
  return v;
}

// Tree drafts ("MTP in TensorRT-LLM on Blackwell", future work: tree
// speculative sampling, Fig. 9): node 0 of a request is the input token and
// node k >= 1 hangs under parents[k] < k. Bit k of a row's path mask is set
// iff node k is on the path from the root to the row's node (itself
// included); a chain (parents == nullptr) gives bits 0..j. A malformed list
// (parents[0] != -1, or some parents[k] outside [0, k)) raises MTP_ERR_TREE
// and yields the chain mask for every row of the request. R <= 16.
__device__ __forceinline__ uint32_t tree_path_mask(const int32_t* parents, int b, int R, int j, unsigned* err) {
  const uint32_t chain = (2u << j) - 1u;
  if (!parents) return chain;
  const int32_t* par = parents + (int64_t)b * R;
  bool ok = par[0] == -1;
  for (int k = 1; k < R; ++k) ok = ok && par[k] >= 0 && par[k] < k;
  if (!ok) {
    raise_error(err, MTP_ERR_TREE);
    return chain;
  }
  uint32_t m = 0;
  for (int k = j; k >= 0; k = par[k]) m |= 1u << k;   // parents decrease: at most j + 1 steps
  return m;
}

// Key t of a request with ctx cached keys is hidden from a row whose path
// mask is m: t is a verify key (t >= ctx) of a node off the row's root path.
__device__ __forceinline__ bool tree_hidden(int t, int ctx, uint32_t m) {
  const int rel = t - ctx;
  return rel >= 0 && (rel >= 32 || ((m >> rel) & 1u) == 0u);
}

// Relaxed acceptance ("MTP in TensorRT-LLM on Blackwell", MTP optimization:
// relaxed acceptance): rank counts of draft d (logit lp) over the logits l of the
// vocabulary entries v a CTA sees: cnt[0] entries ordered before d (larger
// logit, or equal logit and lower id), cnt[1] entries surely above it
// (l > lp + eps), cnt[2] entries that may be above it (l >= lp - eps), with
// eps = kRelaxedRankEps (1 + |lp|). A decision is a near-tie when
// cnt[1] < N <= cnt[2], or when |p_d - (p_1 - delta)| < kRelaxedTieAbs for a
// draft that is not the top-1 token.
constexpr float kRelaxedRankEps = 1e-3f;
constexpr float kRelaxedTieAbs = 1e-3f;

__device__ __forceinline__ void relaxed_count(float l, int v, float lp, int d, float eps, int& before, int& sure,
                                              int& maybe) {
  if (v == d) return;
  before += (l > lp || (l == lp && v < d)) ? 1 : 0;
  sure += l > lp + eps ? 1 : 0;
  maybe += l >= lp - eps ? 1 : 0;
}

// Top-2 of an exponential race: best key k1 at index i1, runner-up key k2.
struct Race {
  float k1;
  int i1;
  float k2;
};

__device__ __forceinline__ Race race_empty() { return Race{-1.0f, -1, -1.0f}; }

__device__ __forceinline__ void race_add(Race& r, float key, int v) {
  // Entries arrive in ascending v within one thread: strict '>' keeps the
  // lowest index among equal keys.
  if (key > r.k1) {
    r.k2 = r.k1;
    r.k1 = key;
    r.i1 = v;
  } else if (key > r.k2) {
    r.k2 = key;
  }
}

__device__ __forceinline__ Race race_merge(Race a, Race b) {
  bool take_b = (b.i1 >= 0) && (a.i1 < 0 || b.k1 > a.k1 || (b.k1 == a.k1 && b.i1 < a.i1));
  Race r;
  if (take_b) {
    r.k1 = b.k1;
    r.i1 = b.i1;
    r.k2 = fmaxf(b.k2, a.k1);
  } else {
    r.k1 = a.k1;
    r.i1 = a.i1;
    r.k2 = fmaxf(a.k2, b.k1);
  }
  return r;
}

__device__ __forceinline__ Race warp_race_merge(Race v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Race w;
    w.k1 = __shfl_xor_sync(0xffffffffu, v.k1, o);
    w.i1 = __shfl_xor_sync(0xffffffffu, v.i1, o);
    w.k2 = __shfl_xor_sync(0xffffffffu, v.k2, o);
    v = race_merge(v, w);
  }
  return v;
}

__device__ __forceinline__ bool race_near_tie(const Race& r) {
  return r.i1 >= 0 && r.k2 >= 0.0f && (r.k1 == r.k2 || r.k1 - r.k2 <= kTieRel * r.k1);
}

}  // namespace mtp
