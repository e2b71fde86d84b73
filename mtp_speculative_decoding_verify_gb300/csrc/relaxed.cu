// Relaxed acceptance ("MTP in TensorRT-LLM on Blackwell", MTP optimization:
// relaxed acceptance): draft d of row j is accepted iff it is among the
// row's N largest logits and p(d) >= p_top1 - delta. The rank is counted
// while the LM head streams the vocabulary; what it needs first is the
// draft's own logit, which this pre-pass computes (one warp per row, a dot
// product of the row's hidden state with the draft's weight row).
#include "common.cuh"
#include "kernels.h"

namespace mtp {

namespace {

constexpr int kThreads = 256;

// dot of two 16-byte vectors of T
__device__ __forceinline__ float dot16(uint4 a, uint4 b, float acc, float) {
  acc = fmaf(__uint_as_float(a.x), __uint_as_float(b.x), acc);
  acc = fmaf(__uint_as_float(a.y), __uint_as_float(b.y), acc);
  acc = fmaf(__uint_as_float(a.z), __uint_as_float(b.z), acc);
  return fmaf(__uint_as_float(a.w), __uint_as_float(b.w), acc);
}
__device__ __forceinline__ float2 bf2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}
__device__ __forceinline__ float dot16(uint4 a, uint4 b, float acc, __nv_bfloat16) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = bf2(av[i]), y = bf2(bv[i]);
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
  }
  return acc;
}
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// lpre[m] = l(m, d_{j+1}) for rows j < D of mode-2 requests, NaN elsewhere
// (NaN marks "no relaxed rank count" for the LM head's epilogue). One CTA
// per row; every thread issues its 16-byte loads of the hidden state and of
// the draft's weight row before using them, so a row costs about one memory
// round trip.
template <typename T>
__global__ void __launch_bounds__(kThreads) relaxed_prepass_kernel(const T* __restrict__ hidden,
                                                                   const T* __restrict__ W,
                                                                   const int32_t* __restrict__ tokens,
                                                                   const uint8_t* __restrict__ mode, int R, int H,
                                                                   int V, float* __restrict__ lpre) {
  __shared__ float s_part[kThreads / 32];
  const int m = blockIdx.x;
  const int b = m / R, j = m % R;
  const int d = j < R - 1 ? tokens[m + 1] : -1;
  if (mode[b] != 2 || d < 0 || d >= V) {
    if (threadIdx.x == 0) lpre[m] = __int_as_float(0x7fc00000);
    return;
  }
  const T* h = hidden + (int64_t)m * H;
  const T* w = W + (int64_t)d * H;
  constexpr int kVec = 16 / sizeof(T);
  float acc = 0.0f;
  const bool vec = H % kVec == 0 && (((uintptr_t)hidden | (uintptr_t)W) & 15) == 0;   // rows 16-byte aligned
  if (vec) {
    const uint4* h4 = reinterpret_cast<const uint4*>(h);
    const uint4* w4 = reinterpret_cast<const uint4*>(w);
    const int nv = H / kVec;
    constexpr int kUnroll = 4;
    for (int i0 = threadIdx.x; i0 < nv; i0 += kThreads * kUnroll) {
      uint4 a[kUnroll], c[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u * kThreads;
        a[u] = i < nv ? __ldg(h4 + i) : make_uint4(0, 0, 0, 0);
        c[u] = i < nv ? __ldg(w4 + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) acc = dot16(a[u], c[u], acc, T());
    }
  } else {
    for (int k = threadIdx.x; k < H; k += kThreads) acc = fmaf(to_f(h[k]), to_f(w[k]), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (threadIdx.x % 32 == 0) s_part[threadIdx.x / 32] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) t += s_part[i];
    lpre[m] = t;
  }
}

}  // namespace

cudaError_t launch_relaxed_prepass(const mtp_lmhead_args& a, const LmPlan& p, cudaStream_t s) {
  if (a.relaxed_topk <= 0 || a.B == 0) return cudaSuccess;
  const int R = a.D + 1;
  float* lpre = (float*)((char*)a.workspace + p.off_lpre);
  if (a.dtype == MTP_F32)
    relaxed_prepass_kernel<float><<<p.M, kThreads, 0, s>>>((const float*)a.hidden, (const float*)a.lm_head,
                                                           a.tokens, a.mode, R, a.H, a.V, lpre);
  else
    relaxed_prepass_kernel<__nv_bfloat16><<<p.M, kThreads, 0, s>>>((const __nv_bfloat16*)a.hidden,
                                                                   (const __nv_bfloat16*)a.lm_head, a.tokens,
                                                                   a.mode, R, a.H, a.V, lpre);
  return cudaGetLastError();
}

}  // namespace mtp
