// Acceptance: merge the LM head's per-slice row statistics, decide how many
// drafts to accept, and draw the correction / bonus token of sampling
// requests.
//
// "MTP principles" §三 stage 3: greedy - a draft is accepted while it equals
// the target argmax, the first mismatch ends the scan; rejection sampling -
// a draft is accepted when P_target/P_draft >= U, otherwise the token is
// redrawn. Stage 4: the step emits 1 .. D+1 tokens, the first rejected
// position replaced by the target's token. "Speculative decoding and MTP"
// §2.3: drafts after the first rejection are dropped whatever their
// probability; §4.4: accept with probability min(1, p/q), and at temperature
// 0 accept only when argmax(p) is the draft, replacing it otherwise.
// "MTP in TensorRT-LLM" Fig. 1: when every draft is accepted the target's
// own next token is accepted too (the bonus). Relaxed requests ("MTP in
// TensorRT-LLM on Blackwell", MTP optimization: relaxed acceptance): a draft
// is accepted while it ranks among the row's relaxed_topk largest logits and
// p(d) >= p(top-1) - relaxed_delta; the first miss is replaced by the argmax.
// Tree drafts ("MTP in TensorRT-LLM on Blackwell", future work: tree
// speculative sampling) are verified greedily edge by edge: a node is
// accepted when its whole root path matches the parents' argmaxes, and the
// deepest accepted node (lowest index on equal depth) ends the emitted path.
//
// The redraw uses the residual max(0, p - q) (normalised) so that the
// emitted tokens follow p exactly; a categorical draw is an exponential race
// argmax_v w_v / E_v with E_v from the Philox stream, so the winner does not
// depend on how the vocabulary is split across CTAs.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace mtp {

namespace {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;

struct Decision {
  int n;         // drafts accepted
  int sampling;  // 1: a race must fill out_tokens[b, n]
  int tie;       // bit0 near-tie of an accept decision
  int pad;
};

}  // namespace

// One CTA per request: reduce the R rows' partials, then warp 0 takes the
// accept decisions in order.
__global__ void __launch_bounds__(kThreads) accept_decide_kernel(
    const float* __restrict__ pmax, const float* __restrict__ psum, const float* __restrict__ pbest,
    const int* __restrict__ pidx, const float* __restrict__ ldraft, int slices, const int32_t* __restrict__ tokens,
    const uint8_t* __restrict__ mode, const float* __restrict__ temperature, const float* __restrict__ q_draft,
    int any_sampling, uint64_t seed, int B, int D, int V, float* __restrict__ ws_lse, int* __restrict__ ws_amax,
    Decision* __restrict__ dec, int* __restrict__ race_count, int32_t* __restrict__ out_tokens,
    int32_t* __restrict__ num_accepted, uint8_t* __restrict__ tie_flags, float* __restrict__ lse_out,
    int32_t* __restrict__ argmax_out, const int* __restrict__ rcnt, int relaxed_topk, float relaxed_delta,
    const int32_t* __restrict__ parents, int32_t* __restrict__ accepted_nodes, unsigned* err) {
  __shared__ float s_lse[kMaxRows];
  __shared__ float s_top[kMaxRows];
  __shared__ int s_amax[kMaxRows];
  __shared__ int s_cnt[kMaxRows][3];
  const int b = blockIdx.x;
  const int R = D + 1;
  const int M = B * R;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int md = mode ? mode[b] : 0;   // no mode array: a draft step (greedy, R = 1)
  const bool relaxed = md == 2 && relaxed_topk > 0;

  for (int j = warp; j < R; j += kWarps) {
    const int m = b * R + j;
    RowStat st = rowstat_empty();
    for (int sl = lane; sl < slices; sl += kWarp) {
      const int64_t o = (int64_t)sl * M + m;
      st = rowstat_merge(st, RowStat{pmax[o], psum[o], pbest[o], pidx[o]});
    }
    st = warp_merge(st);
    if (relaxed && j < D) {   // the draft's rank counts, summed over the LM head's slices
      const int64_t plane = (int64_t)slices * M;
      int c0 = 0, c1 = 0, c2 = 0;
      for (int sl = lane; sl < slices; sl += kWarp) {
        const int64_t o = (int64_t)sl * M + m;
        c0 += rcnt[o];
        c1 += rcnt[plane + o];
        c2 += rcnt[2 * plane + o];
      }
#pragma unroll
      for (int off = kWarp / 2; off > 0; off >>= 1) {
        c0 += __shfl_xor_sync(0xffffffffu, c0, off);
        c1 += __shfl_xor_sync(0xffffffffu, c1, off);
        c2 += __shfl_xor_sync(0xffffffffu, c2, off);
      }
      if (lane == 0) {
        s_cnt[j][0] = c0;
        s_cnt[j][1] = c1;
        s_cnt[j][2] = c2;
      }
    }
    if (lane == 0) {
      const float lse = st.m + logf(st.s);
      s_lse[j] = lse;
      s_top[j] = st.best;
      s_amax[j] = st.idx;
      ws_lse[m] = lse;
      ws_amax[m] = st.idx;
      if (lse_out) lse_out[m] = lse;
      if (argmax_out) argmax_out[m] = st.idx;
    }
  }
  __syncthreads();
  if (threadIdx.x != 0) return;

  const int32_t* tok = tokens ? tokens + (int64_t)b * R : nullptr;   // read only while n < D
  int32_t* out = out_tokens + (int64_t)b * R;
  bool bad = false;
  if (tokens)
    for (int j = 0; j < R; ++j) bad |= (tok[j] < 0 || tok[j] >= V);
  if (bad) raise_error(err, MTP_ERR_TOKEN_ID);
  if (md > 2 || (md == 2 && !relaxed)) raise_error(err, MTP_ERR_MODE);   // decided greedily
  bool sampling = any_sampling && md == 1 && temperature[b] > 0.0f;
  int n = 0, tie = 0;
  // Tree requests: validate the parents list and find the deepest accepted node.
  int tree_end = -1;          // >= 0: the accepted path ends at this node
  int par[kMaxRows];
  if (parents && !bad) {
    if (sampling || md == 2) raise_error(err, MTP_ERR_MODE);   // trees are verified greedily
    sampling = false;
    const int32_t* pb = parents + (int64_t)b * R;
    bool ok = pb[0] == -1;
    int depth[kMaxRows];
    bool acc[kMaxRows];
    depth[0] = 0;
    acc[0] = true;
    int best = 0;
    for (int k = 1; ok && k < R; ++k) {
      const int pk = pb[k];
      ok = pk >= 0 && pk < k;
      if (!ok) break;
      par[k] = pk;
      acc[k] = acc[pk] && tok[k] == s_amax[pk];
      depth[k] = depth[pk] + 1;
      if (acc[k] && depth[k] > depth[best]) best = k;
    }
    if (ok) tree_end = best;
    else raise_error(err, MTP_ERR_TREE);   // verified as a chain
  }
  if (tree_end >= 0) {
    n = 0;
    for (int k = tree_end; k > 0; k = par[k]) ++n;
    // walk back from the end: path node i sits at depth i
    int k = tree_end;
    for (int i = n; i >= 1; --i) {
      out[i - 1] = tok[k];
      if (accepted_nodes) accepted_nodes[(int64_t)b * R + i] = k;
      k = par[k];
    }
    out[n] = s_amax[tree_end];
    for (int j = n + 1; j < R; ++j) out[j] = -1;
    if (accepted_nodes) {
      accepted_nodes[(int64_t)b * R] = 0;
      for (int j = n + 1; j < R; ++j) accepted_nodes[(int64_t)b * R + j] = -1;
    }
  } else if (relaxed && !bad) {
    for (; n < D; ++n) {
      const int d = tok[n + 1];
      const int before = s_cnt[n][0], sure = s_cnt[n][1], maybe = s_cnt[n][2];
      if (sure < relaxed_topk && maybe >= relaxed_topk) tie |= 1;
      const float pd = expf(ldraft[b * R + n] - s_lse[n]);
      const float thr = expf(s_top[n] - s_lse[n]) - relaxed_delta;
      if (d != s_amax[n] && fabsf(pd - thr) < kRelaxedTieAbs) tie |= 1;
      if (!(before < relaxed_topk && pd >= thr)) break;
    }
    for (int j = 0; j < R; ++j) out[j] = j < n ? tok[j + 1] : (j == n ? s_amax[n] : -1);
  } else if (!sampling || bad) {
    while (!bad && n < D && s_amax[n] == tok[n + 1]) ++n;
    for (int j = 0; j < R; ++j) out[j] = j < n ? tok[j + 1] : (j == n ? s_amax[n] : -1);
  } else {
    for (; n < D; ++n) {
      const int x = tok[n + 1];
      const float p = expf(ldraft[b * R + n] - s_lse[n]);
      const float qx = q_draft[((int64_t)b * D + n) * V + x];
      const float u = accept_uniform(seed, (uint32_t)b, (uint32_t)n);
      const float uq = __fmul_rn(u, qx);
      if (qx > 0.0f && fabsf(p - uq) < __fmul_rn(kTieRel, qx)) tie |= 1;
      if (!(p >= uq)) break;
    }
    for (int j = 0; j < R; ++j) out[j] = j < n ? tok[j + 1] : -1;  // out[n] comes from the race
  }
  if (accepted_nodes && tree_end < 0)
    for (int j = 0; j < R; ++j) accepted_nodes[(int64_t)b * R + j] = j <= n ? j : -1;
  dec[b] = Decision{n, (sampling && !bad) ? 1 : 0, tie, 0};
  race_count[b] = 0;
  if (num_accepted) num_accepted[b] = n;
  if (tie_flags) tie_flags[b] = (uint8_t)tie;
}

// Block-wide merge of one race per thread; the result is valid in thread 0.
__device__ __forceinline__ Race block_race_merge(Race r, Race* s_part) {
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  r = warp_race_merge(r);
  __syncthreads();   // s_part may still be read from an earlier merge
  if (lane == 0) s_part[warp] = r;
  __syncthreads();
  if (threadIdx.x == 0)
    for (int w = 1; w < kWarps; ++w) r = race_merge(r, s_part[w]);
  return r;
}

// Grid (B, race_slices): each CTA races one vocabulary slice of the row that
// needs a draw, on the residual weights max(0, p - q) (p itself for the
// bonus row); only entries with positive weight draw their exponential. The
// last CTA of a request to finish merges the slices. If no entry of the row
// has positive weight (p = q everywhere) that CTA races the whole row on p.
__global__ void __launch_bounds__(kThreads) accept_race_kernel(
    const float* __restrict__ samp_logits, const float* __restrict__ q_draft, const float* __restrict__ ws_lse,
    const Decision* __restrict__ dec, Race* __restrict__ parts, int* __restrict__ race_count, uint64_t seed,
    int D, int V, int32_t* __restrict__ out_tokens, uint8_t* __restrict__ tie_flags) {
  __shared__ Race s_part[kWarps];
  __shared__ Race s_win;
  __shared__ int s_last;
  const int b = blockIdx.x;
  const int nsl = gridDim.y, sl_id = blockIdx.y;
  const Decision d = dec[b];
  if (!d.sampling) return;
  const int R = D + 1;
  const int n = d.n;
  const int64_t row = (int64_t)b * R + n;
  const float lse = ws_lse[row];
  const uint32_t tag = n < D ? kTagResidual : kTagBonus;
  const float* lrow = samp_logits + row * V;
  const float* qrow = n < D ? q_draft + ((int64_t)b * D + n) * V : nullptr;
  const int per = ((V + nsl - 1) / nsl + 3) & ~3;   // slices start on 16-byte boundaries of a row
  const int v0 = sl_id * per;
  const int v1 = min(V, v0 + per);

  Race resid = race_empty();
  auto visit = [&](float l, float q, int v) {
    const float w = expf(l - lse) - q;
    if (w > 0.0f) race_add(resid, w / race_exponential(seed, (uint32_t)b, (uint32_t)n, (uint32_t)v, tag), v);
  };
  // Entries 4g .. 4g+3 share one generator call (their race words are the
  // four words of counter (b, n, g, tag)), made only if one of them has a
  // positive weight.
  auto visit4 = [&](const float4& l, const float4& q, int g) {
    const float w[4] = {expf(l.x - lse) - q.x, expf(l.y - lse) - q.y, expf(l.z - lse) - q.z, expf(l.w - lse) - q.w};
    if (!(w[0] > 0.0f || w[1] > 0.0f || w[2] > 0.0f || w[3] > 0.0f)) return;
    const uint4 x = philox4(seed, (uint32_t)b, (uint32_t)n, (uint32_t)g, tag);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (w[k] > 0.0f) race_add(resid, w[k] / race_variate(xs[k]), 4 * g + k);
  };
  if ((V & 3) == 0) {
    // Rows start 16-byte aligned: each thread takes 4 consecutive entries per
    // step (ascending within the thread, as race_add expects) and keeps two
    // steps' loads in flight.
    const float4* l4 = reinterpret_cast<const float4*>(lrow);
    const float4* q4 = reinterpret_cast<const float4*>(qrow);
    const float4 zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int g = v0 / 4 + threadIdx.x; g < v1 / 4; g += 2 * kThreads) {
      const int g2 = g + kThreads;
      const bool two = g2 < v1 / 4;
      const float4 la = __ldg(l4 + g), qa = qrow ? __ldg(q4 + g) : zero;
      const float4 lb = two ? __ldg(l4 + g2) : zero, qb = (two && qrow) ? __ldg(q4 + g2) : zero;
      visit4(la, qa, g);
      if (two) visit4(lb, qb, g2);
    }
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += kThreads) visit(lrow[v], qrow ? qrow[v] : 0.0f, v);
  }
  resid = block_race_merge(resid, s_part);
  if (threadIdx.x == 0) {
    parts[(int64_t)b * nsl + sl_id] = resid;
    __threadfence();
    const int done = atomicAdd(&race_count[b], 1);
    s_last = (done == nsl - 1);
  }
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x == 0) {
    __threadfence();
    const volatile Race* vp = parts + (int64_t)b * nsl;
    Race acc = race_empty();
    for (int sl = 0; sl < nsl; ++sl) acc = race_merge(acc, Race{vp[sl].k1, vp[sl].i1, vp[sl].k2});
    s_win = acc;
  }
  __syncthreads();
  Race win = s_win;
  if (win.i1 < 0) {   // every residual weight is zero: the draw falls back to p
    Race plain = race_empty();
    for (int v = threadIdx.x; v < V; v += kThreads) {
      const float p = expf(lrow[v] - lse);
      if (p > 0.0f) race_add(plain, p / race_exponential(seed, (uint32_t)b, (uint32_t)n, (uint32_t)v, tag), v);
    }
    win = block_race_merge(plain, s_part);
  }
  if (threadIdx.x != 0) return;
  out_tokens[row] = win.i1;
  if (race_near_tie(win)) tie_flags[b] = (uint8_t)(tie_flags[b] | 2);
}

cudaError_t launch_accept(const mtp_lmhead_args& a, const LmPlan& p, unsigned* err, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  char* ws = (char*)a.workspace;
  accept_decide_kernel<<<a.B, kThreads, 0, s>>>(
      (const float*)(ws + p.off_pmax), (const float*)(ws + p.off_psum), (const float*)(ws + p.off_pbest),
      (const int*)(ws + p.off_pidx), (const float*)(ws + p.off_ldraft), p.slices, a.tokens, a.mode, a.temperature,
      a.q_draft, a.any_sampling, a.seed, a.B, a.D, a.V, (float*)(ws + p.off_lse), (int*)(ws + p.off_amax),
      (Decision*)(ws + p.off_dec), (int*)(ws + p.off_count), a.out_tokens, a.num_accepted, a.tie_flags, a.lse_out,
      a.argmax_out, a.relaxed_topk > 0 ? (const int*)(ws + p.off_rcnt) : nullptr, a.relaxed_topk, a.relaxed_delta,
      a.parents, a.accepted_nodes, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !a.any_sampling) return e;
  dim3 grid(a.B, p.race_slices);
  accept_race_kernel<<<grid, kThreads, 0, s>>>((const float*)(ws + p.off_logits), a.q_draft,
                                               (const float*)(ws + p.off_lse), (const Decision*)(ws + p.off_dec),
                                               (Race*)(ws + p.off_race), (int*)(ws + p.off_count), a.seed, a.D,
                                               a.V, a.out_tokens, a.tie_flags);
  return cudaGetLastError();
}

__global__ void rng_debug_kernel(uint64_t seed, uint32_t b, uint32_t j, uint32_t tag, uint32_t v0, int n,
                                 uint32_t* __restrict__ word0, float* __restrict__ race_e,
                                 float* __restrict__ accept_u) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t v = v0 + (uint32_t)i;
  if (word0) word0[i] = philox_word0(seed, b, j, v, tag);
  if (race_e) race_e[i] = race_exponential(seed, b, j, v, tag);
  if (accept_u) accept_u[i] = accept_uniform(seed, b, v);
}

cudaError_t launch_rng_debug(uint64_t seed, uint32_t b, uint32_t j, uint32_t tag, uint32_t v0, int n,
                             uint32_t* word0, float* race_e, float* accept_u, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  rng_debug_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, b, j, tag, v0, n, word0, race_e, accept_u);
  return cudaGetLastError();
}

size_t accept_decision_bytes() { return sizeof(Decision); }
size_t accept_race_part_bytes() { return sizeof(Race); }

}  // namespace mtp
