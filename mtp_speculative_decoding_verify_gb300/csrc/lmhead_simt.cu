// LM head with fused streaming row statistics, CUDA-core (FFMA) version.
// Used for binary32 weights, where tensor-core formats (tf32/bf16) would not
// keep logits within 1e-4 of the exact product.
//
// "Multi Token Prediction" note, K=3 flow step 4: Logits_i = H_i x W_o, all
// verify rows in one product; step 5: softmax over the vocabulary. The
// softmax is never materialised: each CTA owns a contiguous vocabulary range
// and keeps, per row, the running max, the running sum of exp(l - max) and
// the argmax; the accept kernel merges the per-CTA partials. Full logits go
// to memory only for rejection-sampling rows (their residual draw needs the
// whole row once the log-sum-exp is known) and for the optional debug copy.
// Relaxed rows also count the entries that rank before their draft ("MTP in
// TensorRT-LLM on Blackwell", relaxed acceptance; relaxed_count).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

namespace {
constexpr int kTV = 32;   // vocab entries per tile
constexpr int kMR = 64;   // rows per row chunk (blockIdx.y)
constexpr int kKC = 64;   // k-chunk staged in shared memory
constexpr int kThreads = 256;
}  // namespace

template <typename T>
__global__ void __launch_bounds__(kThreads) lmhead_simt_kernel(
    const T* __restrict__ hidden, const T* __restrict__ W, const int32_t* __restrict__ tokens,
    const uint8_t* __restrict__ mode, const float* __restrict__ temperature, int any_sampling, int M, int R, int H,
    int V, int tiles_per_slice, float* __restrict__ pmax, float* __restrict__ psum, float* __restrict__ pbest,
    int* __restrict__ pidx, float* __restrict__ ldraft, float* __restrict__ samp_logits,
    float* __restrict__ logits_debug, const float* __restrict__ lpre, int* __restrict__ rcnt, int slices) {
  __shared__ float Hs[kMR][kKC + 1];
  __shared__ float Ws[kTV][kKC + 1];
  __shared__ float Lt[kMR][kTV + 1];
  __shared__ float s_inv_t[kMR];
  __shared__ int s_draft[kMR];
  __shared__ int s_samp[kMR];
  __shared__ float s_lpre[kMR];

  const int tid = threadIdx.x;
  const int slice = blockIdx.x;
  const int row0 = blockIdx.y * kMR;
  const int ntiles = (V + kTV - 1) / kTV;
  const int tile0 = slice * tiles_per_slice;
  const int tile1 = min(ntiles, tile0 + tiles_per_slice);

  if (tid < kMR) {
    const int m = row0 + tid;
    float inv_t = 1.0f;
    int draft = -1, samp = 0;
    if (m < M) {
      const int b = m / R, j = m % R;
      if (any_sampling && mode[b] == 1 && temperature[b] > 0.0f) {
        inv_t = 1.0f / temperature[b];
        samp = 1;
      }
      if (j < R - 1) draft = tokens[m + 1];
    }
    s_inv_t[tid] = inv_t;
    s_draft[tid] = draft;
    s_samp[tid] = samp;
    s_lpre[tid] = (lpre && m < M) ? lpre[m] : __int_as_float(0x7fc00000);
  }
  RowStat st = rowstat_empty();
  int cnt0 = 0, cnt1 = 0, cnt2 = 0;   // relaxed rank counts of the row of thread tid

  const int c = tid % kWarp;        // vocab column of this thread
  const int rbase = tid / kWarp;    // rows rbase + 8 i
  for (int tile = tile0; tile < tile1; ++tile) {
    const int v0 = tile * kTV;
    float acc[kMR / 8];
#pragma unroll
    for (int i = 0; i < kMR / 8; ++i) acc[i] = 0.0f;
    for (int k0 = 0; k0 < H; k0 += kKC) {
      __syncthreads();
      for (int e = tid; e < kMR * kKC; e += kThreads) {
        const int r = e / kKC, k = e % kKC;
        const int m = row0 + r;
        Hs[r][k] = (m < M && k0 + k < H) ? Num<T>::to_f(hidden[(int64_t)m * H + k0 + k]) : 0.0f;
      }
      for (int e = tid; e < kTV * kKC; e += kThreads) {
        const int r = e / kKC, k = e % kKC;
        const int v = v0 + r;
        Ws[r][k] = (v < V && k0 + k < H) ? Num<T>::to_f(W[(int64_t)v * H + k0 + k]) : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kMR / 8; ++i) {
        if (row0 + rbase + 8 * i < M) {
          float a = acc[i];
#pragma unroll 16
          for (int k = 0; k < kKC; ++k) a = fmaf(Hs[rbase + 8 * i][k], Ws[c][k], a);
          acc[i] = a;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kMR / 8; ++i) {
      const int r = rbase + 8 * i;
      Lt[r][c] = s_samp[r] ? __fmul_rn(acc[i], s_inv_t[r]) : acc[i];
    }
    __syncthreads();
    // Per-row statistics: thread r scans its row's tile in ascending vocab order.
    if (tid < kMR && row0 + tid < M) {
      const int nv = min(kTV, V - v0);
      float cmax = -INFINITY;
      int cidx = 0;
      for (int x = 0; x < nv; ++x) {
        const float l = Lt[tid][x];
        if (l > cmax) {
          cmax = l;
          cidx = x;
        }
      }
      float csum = 0.0f;
      for (int x = 0; x < nv; ++x) csum += expf(Lt[tid][x] - cmax);
      st = rowstat_merge(st, RowStat{cmax, csum, cmax, v0 + cidx});
      const int d = s_draft[tid];
      if (d >= v0 && d < v0 + nv) ldraft[row0 + tid] = Lt[tid][d - v0];
      const float lp = s_lpre[tid];
      if (lp == lp) {   // relaxed row
        const float eps = kRelaxedRankEps * (1.0f + fabsf(lp));
        for (int x = 0; x < nv; ++x) relaxed_count(Lt[tid][x], v0 + x, lp, d, eps, cnt0, cnt1, cnt2);
      }
    }
    // Rows that sample (and the optional debug copy) keep the full logits.
    for (int e = tid; e < kMR * kTV; e += kThreads) {
      const int r = e / kTV, x = e % kTV;
      const int m = row0 + r, v = v0 + x;
      if (m < M && v < V) {
        if (s_samp[r] && samp_logits) samp_logits[(int64_t)m * V + v] = Lt[r][x];
        if (logits_debug) logits_debug[(int64_t)m * V + v] = Lt[r][x];
      }
    }
  }
  if (tid < kMR && row0 + tid < M) {
    const int64_t o = (int64_t)slice * M + row0 + tid;
    pmax[o] = st.m;
    psum[o] = st.s;
    pbest[o] = st.best;
    pidx[o] = st.idx;
    if (rcnt) {
      const int64_t plane = (int64_t)slices * M;
      rcnt[o] = cnt0;
      rcnt[plane + o] = cnt1;
      rcnt[2 * plane + o] = cnt2;
    }
  }
}

cudaError_t launch_lmhead_simt(const mtp_lmhead_args& a, const LmPlan& p, unsigned* err, cudaStream_t s) {
  (void)err;
  const int R = a.D + 1;
  const int ntiles = (a.V + kTV - 1) / kTV;
  const int tps = (ntiles + p.slices - 1) / p.slices;
  dim3 grid(p.slices, (p.M + kMR - 1) / kMR);
  char* ws = (char*)a.workspace;
  float* samp = a.any_sampling ? (float*)(ws + p.off_logits) : nullptr;
#define MTP_SIMT_ARGS                                                                                          \
  a.tokens, a.mode, a.temperature, a.any_sampling, p.M, R, a.H, a.V, tps, (float*)(ws + p.off_pmax),          \
      (float*)(ws + p.off_psum), (float*)(ws + p.off_pbest), (int*)(ws + p.off_pidx), (float*)(ws + p.off_ldraft), \
      samp, a.logits_debug, a.relaxed_topk > 0 ? (const float*)(ws + p.off_lpre) : nullptr,                     \
      a.relaxed_topk > 0 ? (int*)(ws + p.off_rcnt) : nullptr, p.slices
  if (a.dtype == MTP_F32)
    lmhead_simt_kernel<float><<<grid, kThreads, 0, s>>>((const float*)a.hidden, (const float*)a.lm_head,
                                                        MTP_SIMT_ARGS);
  else
    lmhead_simt_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>((const __nv_bfloat16*)a.hidden,
                                                                (const __nv_bfloat16*)a.lm_head, MTP_SIMT_ARGS);
#undef MTP_SIMT_ARGS
  return cudaGetLastError();
}

int lmhead_simt_slices(int V, int sm_count) {
  const int ntiles = (V + kTV - 1) / kTV;
  int slices = std::min(ntiles, 2 * sm_count);
  const int tps = (ntiles + slices - 1) / slices;
  return (ntiles + tps - 1) / tps;
}

}  // namespace mtp
