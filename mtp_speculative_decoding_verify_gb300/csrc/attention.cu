// Verify attention: KV append, SIMT attention (fp32 path), split combine.
//
// "Multi Token Prediction" note, overall flow for K=3 draft tokens, step 2:
// the verify tokens' queries are batched against the reused KV cache and
// every verify token's new K/V is written to the cache for the tokens after
// it. "MTP in TensorRT-LLM", attention for MTP: with K+1 chained input
// tokens a causal mask is all the attention kernel needs. Row j of a request
// with ctx cached tokens therefore attends slots 0 .. ctx+j. With tree drafts
// ("MTP in TensorRT-LLM on Blackwell", future work) row j attends the context
// and the slots of the nodes on its root path instead (tree_path_mask).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

// ------------------------------------------------------------------- append
// Copy n elements, 16 bytes per access when both rows allow it.
template <typename T>
__device__ __forceinline__ void copy_row(const T* __restrict__ src, T* __restrict__ dst, int n) {
  const int bytes = n * (int)sizeof(T);
  if ((bytes % 16) == 0 && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int e = threadIdx.x; e < bytes / 16; e += blockDim.x) d4[e] = s4[e];
  } else {
    for (int e = threadIdx.x; e < n; e += blockDim.x) dst[e] = src[e];
  }
}

// One CTA per (request, verify token): copy that token's K (and V) rows into
// slot ctx+j of the paged cache.
template <typename T>
__global__ void kv_append_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ k_cache,
                                 T* __restrict__ v_cache, const int32_t* __restrict__ block_table,
                                 const int32_t* __restrict__ ctx_lens, int R, int Hkv, int d_qk, int d_v,
                                 int max_blocks, int num_blocks, unsigned* err) {
  const int b = blockIdx.x / R, j = blockIdx.x % R;
  const int ctx = ctx_lens[b];
  if (ctx < 0) {
    if (threadIdx.x == 0) raise_error(err, MTP_ERR_LENGTH);
    return;
  }
  const int slot = ctx + j;
  const int page = slot / kBlock;
  if (page >= max_blocks) {
    if (threadIdx.x == 0) raise_error(err, MTP_ERR_LENGTH);
    return;
  }
  const int blk = block_table[(int64_t)b * max_blocks + page];
  if (blk < 0 || blk >= num_blocks) {
    if (threadIdx.x == 0) raise_error(err, MTP_ERR_BLOCK_ID);
    return;
  }
  const int64_t cache_row = (int64_t)blk * kBlock + (slot % kBlock);
  const int nk = Hkv * d_qk;
  copy_row(k_new + ((int64_t)b * R + j) * nk, k_cache + cache_row * nk, nk);
  if (v_new != nullptr) {
    const int nv = Hkv * d_v;
    copy_row(v_new + ((int64_t)b * R + j) * nv, v_cache + cache_row * nv, nv);
  }
}

cudaError_t launch_kv_append(const mtp_attn_args& a, unsigned* err, cudaStream_t s) {
  const int R = a.D + 1;
  const int Hkv = a.is_mla ? 1 : a.Hkv;
  dim3 grid(a.B * R);
  if (a.B == 0) return cudaSuccess;
  if (a.dtype == MTP_F32) {
    kv_append_kernel<float><<<grid, 128, 0, s>>>((const float*)a.k_new, (const float*)a.v_new, (float*)a.k_cache,
                                                (float*)a.v_cache, a.block_table, a.ctx_lens, R, Hkv, a.d_qk, a.d_v,
                                                a.max_blocks, a.num_blocks, err);
  } else {
    using bf = __nv_bfloat16;
    kv_append_kernel<bf><<<grid, 128, 0, s>>>((const bf*)a.k_new, (const bf*)a.v_new, (bf*)a.k_cache,
                                             (bf*)a.v_cache, a.block_table, a.ctx_lens, R, Hkv, a.d_qk, a.d_v,
                                             a.max_blocks, a.num_blocks, err);
  }
  return cudaGetLastError();
}

// --------------------------------------------------------------------- plan
static int rows_per_cta(const mtp_attn_args& a) {
  if (a.dtype == MTP_F32) return 8;     // SIMT: one warp per row, 8 warps
  if (a.is_mla) return 64;              // MLA tensor-core tile
  return 128;                           // GQA tensor-core CTA: all rows of a KV head (up to 128)
}

AttnPlan plan_attention(const mtp_attn_args& a, int sm_count) {
  AttnPlan p{};
  p.sm_count = sm_count;
  const int R = a.D + 1;
  const int group = a.Hq / a.Hkv;
  p.rows_per_kv = group * R;
  const int row_tiles = (p.rows_per_kv + rows_per_cta(a) - 1) / rows_per_cta(a);
  const int max_len = a.max_blocks * kBlock;
  const long long base = (long long)a.B * (a.is_mla ? 1 : a.Hkv) * row_tiles;
  const int kMinSplitLen = 256;
  int n;
  if (attention_uses_mla_tc(a)) {
    // MLA tiles are long and dispatched longest first: split only until the
    // (request, row block) CTAs fill one wave, since every split adds a
    // partial write and the combine pass. Keys per split <= 8192.
    n = base >= sm_count ? 1 : (int)((sm_count + base - 1) / std::max<long long>(base, 1));
    n = std::max(n, (max_len + 8191) / 8192);
  } else if (a.dtype == MTP_BF16 && attention_mma_supported(a)) {
    // GQA/MHA tensor-core CTAs (mma.sync, or tcgen05 for 49..64 rows per KV
    // head, one CTA per SM in both): take the split count with the
    // shortest estimated time for requests of max_len keys, i.e. waves of
    // CTAs x (keys per split + a CTA's start-up, about 256 keys' worth), plus,
    // once split, the partial outputs' round trip (2 R group n fp32 rows of
    // d_v against the KV bytes, about 2 R group n / max_len of them) and the
    // combine pass (about 256 keys' worth). At least enough splits to give
    // every SM two CTAs (mma.sync; one for tcgen05) when the batch alone does not; splits hold at most
    // 16384 keys so that long requests in a mixed batch leave a short tail.
    const int kMaxSplitLen = 16384, kStartKeys = 256;
    const int per_sm = attention_uses_gqa_tc(a) ? 1 : 2;
    const int fill = (int)std::max<long long>(1, (per_sm * sm_count + base - 1) / std::max<long long>(base, 1));
    const int c0 = std::max(fill, (max_len + kMaxSplitLen - 1) / kMaxSplitLen);
    const int c1 = std::max(c0, std::min(64, (max_len + kMinSplitLen - 1) / kMinSplitLen));
    double best = 0.0;
    n = c0;
    for (int c = c0; c <= c1; ++c) {
      const int sl = ((max_len + c - 1) / c + kBlock - 1) / kBlock * kBlock;
      const int ce = (max_len + sl - 1) / sl;
      const long long waves = (base * ce + sm_count - 1) / sm_count;
      double cost = (double)waves * (sl + kStartKeys);
      if (ce > 1) cost = cost * (1.0 + 2.0 * R * group * ce / max_len) + 256.0;
      if (c == c0 || cost < best) {
        best = cost;
        n = ce;
      }
    }
  } else {
    const int kMaxSplitLen = 4096;
    n = (int)std::max<long long>(1, (2LL * sm_count + base - 1) / std::max<long long>(base, 1));
    n = std::max(n, (max_len + kMaxSplitLen - 1) / kMaxSplitLen);
  }
  n = std::min(n, std::max(1, (max_len + kMinSplitLen - 1) / kMinSplitLen));
  int split_len = (max_len + n - 1) / n;
  // tcgen05 MLA and GQA tiles are 128 keys
  const int gran = (a.is_mla && a.dtype == MTP_BF16) || attention_uses_gqa_tc(a) ? 128 : kBlock;
  split_len = (split_len + gran - 1) / gran * gran;
  p.split_len = split_len;
  p.n_splits = (max_len + split_len - 1) / split_len;
  p.ws_bytes = 0;
  if (p.n_splits > 1) {
    const size_t rows = (size_t)a.B * R * a.Hq;
    p.ws_partial_o = 0;
    p.ws_partial_lse = rows * p.n_splits * a.d_v * sizeof(float);
    p.ws_bytes = p.ws_partial_lse + rows * p.n_splits * sizeof(float);
    p.ws_bytes = (p.ws_bytes + 255) / 256 * 256;
  }
  if (attention_uses_mla_tc(a) || attention_uses_gqa_tc(a)) {   // one int per work item at most
    p.ws_order = p.ws_bytes;
    const size_t items = (size_t)p.n_splits * a.B * row_tiles * (a.is_mla ? 1 : a.Hkv);
    p.ws_bytes += (items * sizeof(int32_t) + 255) / 256 * 256;
  } else if (!a.is_mla && a.dtype == MTP_BF16 && attention_mma_supported(a)) {   // mma.sync GQA: its CTA order
    p.ws_order = p.ws_bytes;
    const size_t items = (size_t)p.n_splits * a.B * a.Hkv * attention_mma_row_tiles(a);
    p.ws_bytes += (items * sizeof(int32_t) + 255) / 256 * 256;
  }
  return p;
}

// -------------------------------------------------------------------- SIMT
// One warp per query row; lane l holds elements l, l+32, ... of q and of the
// running output. Online softmax over the keys of this CTA's split.
template <typename T, int EQ, int EV>
__global__ void __launch_bounds__(256) attention_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k_cache, const T* __restrict__ v_cache,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ ctx_lens, T* __restrict__ out,
    float* __restrict__ part_o, float* __restrict__ part_lse, int R, int Hq, int Hkv, int group, int max_blocks,
    int num_blocks, int split_len, int n_splits, int is_mla, float sm_scale, const int32_t* __restrict__ parents,
    unsigned* err) {
  constexpr int DQ = EQ * kWarp, DV = EV * kWarp;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int split = blockIdx.x;
  const int b = blockIdx.y / Hkv, kvh = blockIdx.y % Hkv;
  const int r = blockIdx.z * (blockDim.x / kWarp) + warp;
  if (r >= group * R) return;
  const int j = r / group, h = kvh * group + r % group;
  const int ctx = ctx_lens[b];
  const int L = ctx + j + 1;
  if (ctx < 0 || ctx + R > max_blocks * kBlock) {
    if (lane == 0 && split == 0) raise_error(err, MTP_ERR_LENGTH);
    return;
  }
  const int t0 = split * split_len;
  if (t0 >= L) return;
  const int t1 = min(L, t0 + split_len);
  const uint32_t path = tree_path_mask(parents, b, R, j, err);   // visible verify keys of this row

  const int64_t row = ((int64_t)b * R + j) * Hq + h;
  float qv[EQ];
#pragma unroll
  for (int i = 0; i < EQ; ++i) qv[i] = Num<T>::to_f(q[row * DQ + i * kWarp + lane]) * sm_scale;
  float acc[EV];
#pragma unroll
  for (int i = 0; i < EV; ++i) acc[i] = 0.0f;
  float m = -INFINITY, l = 0.0f;
  const int kv_heads = is_mla ? 1 : Hkv;
  const int32_t* tbl = block_table + (int64_t)b * max_blocks;
  for (int t = t0; t < t1; ++t) {
    if (tree_hidden(t, ctx, path)) continue;
    const int blk = tbl[t / kBlock];
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) raise_error(err, MTP_ERR_BLOCK_ID);
      continue;
    }
    const int64_t slot = (int64_t)blk * kBlock + (t % kBlock);
    const T* kp = k_cache + (slot * kv_heads + (is_mla ? 0 : kvh)) * DQ;
    float dot = 0.0f;
#pragma unroll
    for (int i = 0; i < EQ; ++i) dot += qv[i] * Num<T>::to_f(kp[i * kWarp + lane]);
    const float sc = warp_sum(dot);
    const float m_new = fmaxf(m, sc);
    const float corr = expf(m - m_new);
    const float pr = expf(sc - m_new);
    l = l * corr + pr;
    const T* vp = is_mla ? kp : v_cache + (slot * kv_heads + kvh) * DV;
#pragma unroll
    for (int i = 0; i < EV; ++i) acc[i] = acc[i] * corr + pr * Num<T>::to_f(vp[i * kWarp + lane]);
    m = m_new;
  }
  const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
  if (n_splits == 1) {
#pragma unroll
    for (int i = 0; i < EV; ++i) out[row * DV + i * kWarp + lane] = Num<T>::from_f(acc[i] * inv_l);
  } else {
    float* po = part_o + (row * n_splits + split) * DV;
#pragma unroll
    for (int i = 0; i < EV; ++i) po[i * kWarp + lane] = acc[i] * inv_l;
    if (lane == 0) part_lse[row * n_splits + split] = m + logf(l);
  }
}

template <typename T, int EQ, int EV>
static void run_simt(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s) {
  const int R = a.D + 1, group = a.Hq / a.Hkv;
  const int kv_heads = a.is_mla ? 1 : a.Hkv;
  dim3 grid(p.n_splits, a.B * kv_heads, (group * R + 7) / 8);
  float* po = p.n_splits > 1 ? (float*)((char*)a.workspace + p.ws_partial_o) : nullptr;
  float* pl = p.n_splits > 1 ? (float*)((char*)a.workspace + p.ws_partial_lse) : nullptr;
  attention_simt_kernel<T, EQ, EV><<<grid, 256, 0, s>>>(
      (const T*)a.q, (const T*)a.k_cache, (const T*)a.v_cache, a.block_table, a.ctx_lens, (T*)a.out, po, pl, R,
      a.Hq, kv_heads, group, a.max_blocks, a.num_blocks, p.split_len, p.n_splits, a.is_mla, a.sm_scale, a.parents,
      err);
}

cudaError_t launch_attention_simt(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  using bf = __nv_bfloat16;
  if (a.dtype == MTP_F32) {
    if (a.d_qk == 64 && a.d_v == 64) run_simt<float, 2, 2>(a, p, err, s);
    else if (a.d_qk == 128 && a.d_v == 128) run_simt<float, 4, 4>(a, p, err, s);
    else return cudaErrorInvalidValue;
  } else {
    if (a.is_mla && a.d_qk == 576 && a.d_v == 512) run_simt<bf, 18, 16>(a, p, err, s);
    else if (a.d_qk == 64 && a.d_v == 64) run_simt<bf, 2, 2>(a, p, err, s);
    else if (a.d_qk == 128 && a.d_v == 128) run_simt<bf, 4, 4>(a, p, err, s);
    else return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ combine
// One warp per (request, row, head): merge the non-empty splits with
// weights exp(lse_s - LSE). The warp first turns the splits' log-sum-exps
// into weights (one split per lane), then each lane sums its 4 output
// elements over the splits with 16-byte loads, several splits in flight.
constexpr int kCombineThreads = 256;
constexpr int kCombineMaxSplits = 64;   // weights kept in shared memory up to this many splits

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&lo);
  u.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = u;
}

template <typename T>
__global__ void __launch_bounds__(kCombineThreads) attention_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse, const int32_t* __restrict__ ctx_lens,
    T* __restrict__ out, int B, int R, int Hq, int d_v, int split_len, int n_splits, int max_len) {
  __shared__ float s_w[kCombineThreads / kWarp][kCombineMaxSplits];
  const int wl = threadIdx.x / kWarp;
  const int warp = blockIdx.x * (kCombineThreads / kWarp) + wl, lane = threadIdx.x % kWarp;
  const int rows = B * R * Hq;
  if (warp >= rows) return;
  const int b = warp / (R * Hq), j = (warp / Hq) % R;
  const int ctx = ctx_lens[b];
  if (ctx < 0 || ctx + R > max_len) return;
  const int L = ctx + j + 1;
  const int ns = min(n_splits, (L + split_len - 1) / split_len);
  const float* lse = part_lse + (int64_t)warp * n_splits;
  float mx = -INFINITY;
  for (int sp = lane; sp < ns; sp += kWarp) mx = fmaxf(mx, lse[sp]);
#pragma unroll
  for (int o = kWarp / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float denom = 0.0f;
  for (int sp = lane; sp < ns; sp += kWarp) {
    const float w = expf(lse[sp] - mx);
    if (sp < kCombineMaxSplits) s_w[wl][sp] = w;
    denom += w;
  }
#pragma unroll
  for (int o = kWarp / 2; o > 0; o >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, o);
  __syncwarp();
  const float inv = 1.0f / denom;
  const float* po = part_o + (int64_t)warp * n_splits * d_v;
  T* dst = out + (int64_t)warp * d_v;
  if ((d_v & 3) == 0 && ns <= kCombineMaxSplits) {
    for (int e = 4 * lane; e < d_v; e += 4 * kWarp) {
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 8
      for (int sp = 0; sp < ns; ++sp) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(po + (int64_t)sp * d_v + e));
        const float w = s_w[wl][sp];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
      store4<T>(dst + e, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
  } else {   // many splits or an odd width: weights recomputed per split
    for (int e = lane; e < d_v; e += kWarp) {
      float acc = 0.0f;
      for (int sp = 0; sp < ns; ++sp) acc += expf(lse[sp] - mx) * po[(int64_t)sp * d_v + e];
      dst[e] = Num<T>::from_f(acc * inv);
    }
  }
}

cudaError_t launch_attention_combine(const mtp_attn_args& a, const AttnPlan& p, cudaStream_t s) {
  if (p.n_splits == 1 || a.B == 0) return cudaSuccess;
  const int R = a.D + 1;
  const int rows = a.B * R * a.Hq;
  const int threads = kCombineThreads;
  const int blocks = (rows * kWarp + threads - 1) / threads;
  const float* po = (const float*)((const char*)a.workspace + p.ws_partial_o);
  const float* pl = (const float*)((const char*)a.workspace + p.ws_partial_lse);
  if (a.dtype == MTP_F32)
    attention_combine_kernel<float><<<blocks, threads, 0, s>>>(po, pl, a.ctx_lens, (float*)a.out, a.B, R, a.Hq,
                                                               a.d_v, p.split_len, p.n_splits, a.max_blocks * kBlock);
  else
    attention_combine_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(po, pl, a.ctx_lens, (__nv_bfloat16*)a.out,
                                                                       a.B, R, a.Hq, a.d_v, p.split_len, p.n_splits,
                                                                       a.max_blocks * kBlock);
  return cudaGetLastError();
}

}  // namespace mtp
