// Verify attention on bf16 tensor cores: paged KV tiles staged by TMA into a
// shared-memory ring (one producer warp), QK^T and PV with mma.sync
// m16n8k16 (fp32 accumulate), online softmax in registers with quad
// shuffles. Split-KV partials are merged by attention_combine_kernel.
//
// "Multi Token Prediction" note, K=3 flow step 2: the verify tokens' queries
// are stacked into one Q matrix against the reused cache, and each verify
// token sees the K/V of the tokens before it plus its own; "MTP in
// TensorRT-LLM", attention for MTP: K+1 chained queries need only a causal
// mask. Row of verify token j (request context ctx) attends slots 0..ctx+j.
//
// attn_gqa_kernel<D, tree, form>: GQA/MHA, d_qk = d_v = D (64 or 128). CTA =
// (split, request x KV head, row block): the g*R query rows that share one
// KV head (up to 112: one row warp per 16 rows), 64-key tiles = one cache
// block. CTAs take their work items longest first from an order computed
// just before the launch (gqa_mma_schedule_kernel). Forms 1 and 2 add key parts: warps sharing rows take alternate tiles
// and merge their softmax state at the end (see run_gqa). Tree drafts use a
// per-row root-path mask instead of the causal limit. (Absorbed MLA runs on
// tcgen05: attention_mla_tc.cu.)
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"
#include "sm100.cuh"

namespace mtp {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box);

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnKParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* part_o;
  float* part_lse;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* parents;        // [B, R] tree drafts, nullptr: chains
  unsigned* err;
  int R, Hq, Hkv, group, rows;  // rows = query rows per (request, KV head)
  int row_warps, key_parts;     // consumer warps = row_warps x key_parts (warps sharing rows split the tiles)
  int max_blocks, num_blocks, split_len, n_splits, stages;
  int B, row_tiles;              // requests, CTAs per (split, request, KV head)
  const int32_t* order;          // CTA -> work item, longest first (gqa_mma_schedule_kernel)
  float scale_log2;              // sm_scale * log2(e)
};

// ------------------------------------------------------------------ GQA
constexpr int kGqaRowsPerCta = 112;   // up to 7 row warps x 16 rows
// Consumers (row warps x key parts) + 1 producer warp: 7 consumers keep the
// 8 warps at 2 per SM sub-partition (up to 255 registers a thread); the wide
// form with 8 consumers (4 row warps x 2 key parts) puts 3 warps on one
// sub-partition and so has at most 168 registers a thread.
constexpr int kGqaConsumers = 7, kGqaConsumersWide = 8;
// The narrow form: at most 3 row warps (48 rows) and no key parts, compiled
// for three CTAs per SM (at most 170 registers a thread), so that three CTAs
// of two stages each share an SM instead of two of three stages.
constexpr int kGqaConsumersNarrow = 3;

template <int D>
struct GqaCfg {
  static constexpr int kTileKeys = 64;                         // one cache block
  static constexpr int kBox = kTileKeys * 128;                 // bytes of one [64 keys][64 dims] box
  static constexpr int kKBytes = (D / 64) * kBox;
  static constexpr int kStageBytes = 2 * kKBytes;              // K and V
};

// kTree: rows see the verify keys of their root path (tree drafts) instead of
// a causal prefix; the chain instantiation keeps the plain limit test.
// kForm: 0 one warp per 16 rows, each reading every tile (the loop keeps a
// running stage / phase); 1 key parts on up to 7 consumers; 2 the wide form,
// 8 consumers; 3 form 0 for at most 3 row warps at three CTAs per SM.
template <int D, bool kTree, int kForm>
__global__ void __launch_bounds__(kForm == 3 ? 32 * (kGqaConsumersNarrow + 1)
                                             : 32 * ((kForm == 2 ? kGqaConsumersWide : kGqaConsumers) + 1),
                                  kForm == 3 ? 3 : 1) attn_gqa_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                       const __grid_constant__ CUtensorMap tm_v,
                                                       const AttnKParams p) {
  using C = GqaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * C::kStageBytes);
  uint64_t* empty = full + p.stages;
  int* stage_valid = reinterpret_cast<int*>(empty + p.stages);
  volatile int* abort = stage_valid + p.stages;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_cons = blockDim.x / 32 - 1;
  // Work item of this CTA: ((split * B + b) * Hkv + kvh) * row_tiles + row tile.
  const int item = p.order[blockIdx.x];
  const int per = p.Hkv * p.row_tiles;
  const int split = item / (per * p.B);
  const int b = (item / per) % p.B;
  const int kvh = (item % per) / p.row_tiles;
  const int row_base = (item % p.row_tiles) * kGqaRowsPerCta;
  const int ctx = p.ctx_lens[b];
  if (ctx < 0 || ctx + p.R > p.max_blocks * kBlock) {
    if (threadIdx.x == 0 && split == 0) raise_error(p.err, MTP_ERR_LENGTH);
    return;
  }
  const int t0 = split * p.split_len;
  const int t_end = min(t0 + p.split_len, ctx + p.R);   // keys this CTA may need
  if (t0 >= t_end) return;
  const int page0 = t0 / C::kTileKeys;
  const int n_tiles = (t_end - t0 + C::kTileKeys - 1) / C::kTileKeys;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      sm100::mbar_init(&full[s], 1);
      sm100::mbar_init(&empty[s], p.row_warps);   // every tile is read by one warp per row block
    }
    *abort = 0;
    sm100::fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      sm100::tma_prefetch_desc(&tm_k);
      sm100::tma_prefetch_desc(&tm_v);
      const uint64_t pol = sm100::l2_policy_evict_first();
      const int32_t* tbl = p.block_table + (int64_t)b * p.max_blocks;
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[8];
      for (int s2 = 0; s2 < 8; ++s2) last_parity[s2] = -1;
      for (int i = 0; i < n_tiles; ++i) {
        if (!sm100::mbar_wait(&empty[stage], phase ^ 1u, abort)) {
          *abort = 1;
          raise_error(p.err, MTP_ERR_TIMEOUT);
          break;
        }
        const int blk = tbl[page0 + i];
        const bool valid = blk >= 0 && blk < p.num_blocks;
        stage_valid[stage] = valid ? 1 : 0;
        uint8_t* ks = smem + stage * C::kStageBytes;
        if (valid) {
          sm100::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            sm100::tma_load_4d(ks + c * C::kBox, &tm_k, &full[stage], c * 64, kvh, 0, blk, pol);
            sm100::tma_load_4d(ks + C::kKBytes + c * C::kBox, &tm_v, &full[stage], c * 64, kvh, 0, blk, pol);
          }
          last_parity[stage] = (int)phase;
        } else {
          raise_error(p.err, MTP_ERR_BLOCK_ID);
          sm100::mbar_arrive(&full[stage]);
        }
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Every copy issued must land before the CTA may exit (consumers wait
      // for all of them unless they aborted; this covers the abort case).
      for (int s2 = 0; s2 < p.stages; ++s2)
        if (last_parity[s2] >= 0)
          sm100::mbar_wait_timeout(&full[s2], (uint32_t)last_parity[s2], sm100::kWaitTimeoutNs);
    }
    return;
  }

  // ---------------------------------------------------------- consumers
  // Consumer cw takes rows 16 rw .. 16 rw + 15 of the CTA and the tiles i
  // with i % key_parts == kp; the key parts of a row block merge at the end.
  const int cw = warp - 1;
  constexpr bool kOnePart = kForm == 0 || kForm == 3;   // no key parts
  const int rw = kOnePart ? cw : cw % p.row_warps, kp = kOnePart ? 0 : cw / p.row_warps;
  const int g = lane >> 2, t = lane & 3;
  const int r_lo = row_base + rw * 16 + g, r_hi = r_lo + 8;
  const int rl = min(r_lo, p.rows - 1), rh = min(r_hi, p.rows - 1);   // padding rows compute on the last row
  const int j_lo = rl / p.group, j_hi = rh / p.group;
  const int h_lo = kvh * p.group + rl % p.group, h_hi = kvh * p.group + rh % p.group;
  const int lim_lo = ctx + j_lo, lim_hi = ctx + j_hi;
  const uint32_t path_lo = kTree ? tree_path_mask(p.parents, b, p.R, j_lo, p.err) : 0u;   // visible verify keys
  const uint32_t path_hi = kTree ? tree_path_mask(p.parents, b, p.R, j_hi, p.err) : 0u;
  const int mask_from = kTree ? ctx : min(lim_lo, lim_hi) + 1;   // first key a row may not see
  const int64_t qrow_lo = ((int64_t)b * p.R + j_lo) * p.Hq + h_lo;
  const int64_t qrow_hi = ((int64_t)b * p.R + j_hi) * p.Hq + h_hi;

  // Q fragments (A operand) for all D/16 k-steps, straight from global memory.
  uint32_t qa[D / 16][4];
  {
    const uint32_t* qlo = reinterpret_cast<const uint32_t*>(p.q + qrow_lo * D);
    const uint32_t* qhi = reinterpret_cast<const uint32_t*>(p.q + qrow_hi * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = qlo[(kk * 16 + 2 * t) / 2];
      qa[kk][1] = qhi[(kk * 16 + 2 * t) / 2];
      qa[kk][2] = qlo[(kk * 16 + 8 + 2 * t) / 2];
      qa[kk][3] = qhi[(kk * 16 + 8 + 2 * t) / 2];
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.0f, l_hi = 0.0f;

  // One tile: wait for its stage, S = Q K^T, online softmax, O += P V,
  // release the stage. False when the wait gave up.
  auto consume = [&](int i, int stage, uint32_t phase) -> bool {
    if (!__all_sync(0xffffffffu, sm100::mbar_wait(&full[stage], phase, abort) ? 1 : 0)) {
      if (lane == 0) {
        *abort = 1;
        raise_error(p.err, MTP_ERR_TIMEOUT);
      }
      return false;
    }
    if (stage_valid[stage]) {
      const uint32_t kbase = sm100::smem_u32(smem + stage * C::kStageBytes);
      const uint32_t vbase = kbase + C::kKBytes;
      // S = Q K^T for 16 rows x 64 keys.
      float s[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.0f;
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
          const int dim = kk * 16 + (mi & 1) * 8;
          uint32_t b0, b1, b2, b3;
          mma::ldsm_x4(kbase + mma::sw128_boxed(64, key, dim), b0, b1, b2, b3);
          mma::mma_bf16_16816(s[2 * np], qa[kk], b0, b1);
          mma::mma_bf16_16816(s[2 * np + 1], qa[kk], b2, b3);
        }
      }
      // Scale, causal mask, online softmax (rows r_lo / r_hi).
      const int tk = (page0 + i) * C::kTileKeys;
      const bool need_mask = tk + C::kTileKeys - 1 >= mask_from;
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[n][e] * p.scale_log2;
          if (need_mask) {
            const int key = tk + n * 8 + 2 * t + (e & 1);
            const bool hidden = kTree ? tree_hidden(key, ctx, (e < 2) ? path_lo : path_hi)
                                      : key > ((e < 2) ? lim_lo : lim_hi);
            if (hidden) v = -INFINITY;
          }
          s[n][e] = v;
        }
        mx_lo = fmaxf(mx_lo, fmaxf(s[n][0], s[n][1]));
        mx_hi = fmaxf(mx_hi, fmaxf(s[n][2], s[n][3]));
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float base_lo = mn_lo == -INFINITY ? 0.0f : mn_lo;
      const float base_hi = mn_hi == -INFINITY ? 0.0f : mn_hi;
      const float c_lo = exp2f(m_lo - base_lo), c_hi = exp2f(m_hi - base_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      l_lo *= c_lo;
      l_hi *= c_hi;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= c_lo;
        o[n][1] *= c_lo;
        o[n][2] *= c_hi;
        o[n][3] *= c_hi;
      }
      uint32_t pa[4][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float p0 = exp2f(s[n][0] - base_lo), p1 = exp2f(s[n][1] - base_lo);
        const float p2 = exp2f(s[n][2] - base_hi), p3 = exp2f(s[n][3] - base_hi);
        l_lo += p0 + p1;
        l_hi += p2 + p3;
        pa[n >> 1][(n & 1) * 2 + 0] = mma::pack_bf16(p0, p1);
        pa[n >> 1][(n & 1) * 2 + 1] = mma::pack_bf16(p2, p3);
      }
      // O += P V: k = 64 keys (4 steps), n = D dims.
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int key = kp * 16 + (mi & 1) * 8 + (lane & 7);
          const int dim = dp * 16 + (mi >> 1) * 8;
          uint32_t b0, b1, b2, b3;
          mma::ldsm_x4_trans(vbase + mma::sw128_boxed(64, key, dim), b0, b1, b2, b3);
          mma::mma_bf16_16816(o[2 * dp], pa[kp], b0, b1);
          mma::mma_bf16_16816(o[2 * dp + 1], pa[kp], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(&empty[stage]);
    return true;
  };
  if constexpr (kOnePart) {
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n_tiles; ++i) {
      if (!consume(i, stage, phase)) break;
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else {
    for (int i = kp; i < n_tiles; i += p.key_parts)
      if (!consume(i, i % p.stages, (uint32_t)(i / p.stages) & 1u)) break;
  }

  if constexpr (!kOnePart) {
    // Merge the key parts of each row block. Every consumer is past its last
    // tile at the first barrier, so the stage ring is free: parts kp > 0
    // leave their (o, m, l) there, one slot per (warp, lane) (the fragment
    // layout is the same in every part), and part 0 folds them in.
    constexpr int kVals = D / 2 + 4;
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons * 32) : "memory");
    if (kp > 0) {
      float* xs = reinterpret_cast<float*>(smem) + ((size_t)cw * 32 + lane) * kVals;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        xs[4 * n] = o[n][0];
        xs[4 * n + 1] = o[n][1];
        xs[4 * n + 2] = o[n][2];
        xs[4 * n + 3] = o[n][3];
      }
      xs[D / 2] = m_lo;
      xs[D / 2 + 1] = m_hi;
      xs[D / 2 + 2] = l_lo;
      xs[D / 2 + 3] = l_hi;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons * 32) : "memory");
    if (kp > 0) return;
    for (int q = 1; q < p.key_parts; ++q) {
      const float* ys = reinterpret_cast<const float*>(smem) + ((size_t)(q * p.row_warps + rw) * 32 + lane) * kVals;
      const float mb_lo = ys[D / 2], mb_hi = ys[D / 2 + 1];
      const float mx_lo = fmaxf(m_lo, mb_lo), mx_hi = fmaxf(m_hi, mb_hi);
      const float fa_lo = m_lo == -INFINITY ? 0.0f : exp2f(m_lo - mx_lo);
      const float fb_lo = mb_lo == -INFINITY ? 0.0f : exp2f(mb_lo - mx_lo);
      const float fa_hi = m_hi == -INFINITY ? 0.0f : exp2f(m_hi - mx_hi);
      const float fb_hi = mb_hi == -INFINITY ? 0.0f : exp2f(mb_hi - mx_hi);
      l_lo = l_lo * fa_lo + ys[D / 2 + 2] * fb_lo;
      l_hi = l_hi * fa_hi + ys[D / 2 + 3] * fb_hi;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] = o[n][0] * fa_lo + ys[4 * n] * fb_lo;
        o[n][1] = o[n][1] * fa_lo + ys[4 * n + 1] * fb_lo;
        o[n][2] = o[n][2] * fa_hi + ys[4 * n + 2] * fb_hi;
        o[n][3] = o[n][3] * fa_hi + ys[4 * n + 3] * fb_hi;
      }
      m_lo = mx_lo;
      m_hi = mx_hi;
    }
  }

  // Row sums across the quad, normalise, store.
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float inv_lo = l_lo > 0.0f ? 1.0f / l_lo : 0.0f;
  const float inv_hi = l_hi > 0.0f ? 1.0f / l_hi : 0.0f;
  const bool st_lo = r_lo < p.rows, st_hi = r_hi < p.rows;
  if (p.n_splits == 1) {
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int dim = n * 8 + 2 * t;
      if (st_lo)
        *reinterpret_cast<uint32_t*>(p.out + qrow_lo * D + dim) = mma::pack_bf16(o[n][0] * inv_lo, o[n][1] * inv_lo);
      if (st_hi)
        *reinterpret_cast<uint32_t*>(p.out + qrow_hi * D + dim) = mma::pack_bf16(o[n][2] * inv_hi, o[n][3] * inv_hi);
    }
  } else {
    float* po_lo = p.part_o + (qrow_lo * p.n_splits + split) * D;
    float* po_hi = p.part_o + (qrow_hi * p.n_splits + split) * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int dim = n * 8 + 2 * t;
      if (st_lo) *reinterpret_cast<float2*>(po_lo + dim) = make_float2(o[n][0] * inv_lo, o[n][1] * inv_lo);
      if (st_hi) *reinterpret_cast<float2*>(po_hi + dim) = make_float2(o[n][2] * inv_hi, o[n][3] * inv_hi);
    }
    if (t == 0) {
      if (st_lo) p.part_lse[qrow_lo * p.n_splits + split] = l_lo > 0.0f ? m_lo * kLn2 + logf(l_lo) : -INFINITY;
      if (st_hi) p.part_lse[qrow_hi * p.n_splits + split] = l_hi > 0.0f ? m_hi * kLn2 + logf(l_hi) : -INFINITY;
    }
  }
}


// --------------------------------------------------------------- launchers
template <int D>
int gqa_smem_bytes(int stages) {
  return stages * GqaCfg<D>::kStageBytes + stages * 20 + 64 + 1024;
}

constexpr int kGqaMaxSmem = 232448;   // 227 KB opt-in per CTA

template <int D>
using GqaKernel = void (*)(const CUtensorMap, const CUtensorMap, const AttnKParams);

template <int D>
GqaKernel<D> gqa_kernel(bool tree, int form) {
  if (form == 3) return tree ? attn_gqa_kernel<D, true, 3> : attn_gqa_kernel<D, false, 3>;
  if (form == 2) return tree ? attn_gqa_kernel<D, true, 2> : attn_gqa_kernel<D, false, 2>;
  if (form == 1) return tree ? attn_gqa_kernel<D, true, 1> : attn_gqa_kernel<D, false, 1>;
  return tree ? attn_gqa_kernel<D, true, 0> : attn_gqa_kernel<D, false, 0>;
}

// CTAs of one form that fit on an SM at once (the occupancy the runtime
// reports for its threads and shared memory), cached per form.
template <int D>
int gqa_occupancy(bool tree, int form, int warps, int stages) {
  static int cache[2][4][kGqaConsumersWide + 1][9] = {};
  int& c = cache[tree][form][warps][stages];
  if (c == 0) {
    const GqaKernel<D> kern = gqa_kernel<D>(tree, form);
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGqaMaxSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * (warps + 1), gqa_smem_bytes<D>(stages)) !=
            cudaSuccess)
      n = 1;
    c = std::max(1, n);
  }
  return c;
}

constexpr int kMaxOrderTiles = 256;   // split_len <= 16384 keys = 256 cache blocks

// CTA order of the GQA kernel, longest first (counting sort by the number
// of 64-key tiles, one CTA): the block scheduler starts CTAs in index order,
// so the long splits of long requests start in the first waves and the short
// ones fill the tail, instead of whatever request happens to come last. The
// row tiles and KV heads of one (split, request) stay adjacent: they read the
// same cache pages (the heads of a token are interleaved in a block).
__global__ void __launch_bounds__(1024) gqa_mma_schedule_kernel(const int32_t* __restrict__ ctx_lens, int B, int R,
                                                               int per, int split_len, int n_splits, int max_len,
                                                               int32_t* __restrict__ order) {
  __shared__ int hist[kMaxOrderTiles + 1];
  const int n = n_splits * B;   // groups (split, request); group q = split * B + b holds items q * per + i
  auto tiles_of = [&](int q) -> int {
    const int ctx = ctx_lens[q % B];
    if (ctx < 0 || ctx + R > max_len) return 0;   // the attention kernel reports and skips the request
    const int t0 = (q / B) * split_len;
    const int t_end = min(t0 + split_len, ctx + R);
    return t0 < t_end ? min((t_end - t0 + kBlock - 1) / kBlock, kMaxOrderTiles) : 0;
  };
  for (int k = threadIdx.x; k <= kMaxOrderTiles; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < n; q += blockDim.x) atomicAdd(&hist[tiles_of(q)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {   // hist[k] becomes the first group position of tile count k
    int acc = 0;
    for (int k = kMaxOrderTiles; k >= 0; --k) {
      const int h = hist[k];
      hist[k] = acc;
      acc += h;
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const int pos = atomicAdd(&hist[tiles_of(q)], 1);
    for (int i = 0; i < per; ++i) order[pos * per + i] = q * per + i;
  }
}

template <int D>
cudaError_t run_gqa(const mtp_attn_args& a, const AttnPlan& pl, unsigned* err, cudaStream_t s) {
  // Consumer layout: one warp per 16 rows of the CTA. When a KV head has few
  // rows, spare warps can take alternate tiles of the same rows (key parts)
  // and merge at the end. Tile i sits in stage i % stages and goes to part
  // i % key_parts; stages is a multiple of key_parts, so each stage serves
  // one part, which meets that stage's phases in order (a part that skipped
  // ahead to a stage of another part could take a phase that has not
  // completed for a completed one: the parity wait cannot tell them apart).
  // Key parts are used only when they put more consumer warps on an SM than
  // single-part CTAs do at their occupancy (two of those often share an SM),
  // the grid fills at least two waves of single-part CTAs, and each part gets
  // at least 4 tiles. The wide form (8 consumers) only serves 4 row warps,
  // which 7 consumers cannot split.
  const int R = a.D + 1, group = a.Hq / a.Hkv, rows = group * R;
  const bool tree = a.parents != nullptr;
  constexpr int kMaxStages = 8;   // the producer tracks at most 8 stages
  const int s_max = std::min(kMaxStages, (kGqaMaxSmem - 2048) / GqaCfg<D>::kStageBytes);
  const int row_warps = std::min(kGqaRowsPerCta / 16, (rows + 15) / 16);
  const int max_tiles = (pl.split_len + kBlock - 1) / kBlock;
  const long long grid_ctas =
      (long long)pl.n_splits * a.B * a.Hkv * ((rows + kGqaRowsPerCta - 1) / kGqaRowsPerCta);
  int key_parts = 1, stages = D == 128 ? 3 : 4, form = 0;
  const int occ1 = gqa_occupancy<D>(tree, 0, row_warps, stages);
  if (grid_ctas >= 2LL * occ1 * pl.sm_count) {
    int best = occ1 * row_warps;
    for (int k = 2; k <= s_max && 4 * k <= max_tiles; ++k) {
      const bool w = row_warps * k > kGqaConsumers;
      if (w && !(row_warps == 4 && k == 2)) continue;
      const int S = k * (s_max / k);
      const int cons = gqa_occupancy<D>(tree, w ? 2 : 1, row_warps * k, S) * row_warps * k;
      if (cons > best) {
        best = cons;
        key_parts = k;
        stages = S;
        form = w ? 2 : 1;
      }
    }
  }
  if (form == 0 && row_warps <= kGqaConsumersNarrow) {
    // The same consumers three to an SM (two stages each) when the whole grid
    // then runs in one wave and does not at the register-bound two CTAs of
    // three stages (sweep B=8, D=5: 0.071 -> 0.054 ms). Over several waves the
    // shallower pipeline loses (Llama-70B shape: 0.196 -> 0.216 ms).
    const long long occ0 = gqa_occupancy<D>(tree, 0, row_warps, stages);
    const long long occ3 = gqa_occupancy<D>(tree, 3, row_warps, 2);
    if (occ3 > occ0 && grid_ctas > occ0 * pl.sm_count && grid_ctas <= occ3 * pl.sm_count) {
      form = 3;
      stages = 2;
    }
  }
  const int warps = row_warps * key_parts;
  CUtensorMap tk, tv;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.Hkv, (cuuint64_t)kBlock, (cuuint64_t)a.num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hkv * D * 2, (cuuint64_t)kBlock * a.Hkv * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kBlock, 1};
  if (!make_bf16_map(&tk, a.k_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
  if (!make_bf16_map(&tv, a.v_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
  AttnKParams p;
  p.q = (const __nv_bfloat16*)a.q;
  p.out = (__nv_bfloat16*)a.out;
  p.part_o = pl.n_splits > 1 ? (float*)((char*)a.workspace + pl.ws_partial_o) : nullptr;
  p.part_lse = pl.n_splits > 1 ? (float*)((char*)a.workspace + pl.ws_partial_lse) : nullptr;
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.parents = a.parents;
  p.err = err;
  p.R = R;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = group;
  p.rows = rows;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.stages = stages;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.row_warps = row_warps;
  p.key_parts = key_parts;
  // the merge of the key parts stages every consumer's (o, m, l) in the stage ring
  if ((size_t)warps * 32 * (D / 2 + 4) * sizeof(float) > (size_t)stages * GqaCfg<D>::kStageBytes)
    return cudaErrorInvalidValue;
  const int smem = gqa_smem_bytes<D>(stages);
  const GqaKernel<D> kern = gqa_kernel<D>(tree, form);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  p.B = a.B;
  p.row_tiles = (rows + kGqaRowsPerCta - 1) / kGqaRowsPerCta;
  int32_t* order = (int32_t*)((char*)a.workspace + pl.ws_order);
  p.order = order;
  const int per = a.Hkv * p.row_tiles;
  gqa_mma_schedule_kernel<<<1, 1024, 0, s>>>(a.ctx_lens, a.B, R, per, pl.split_len, pl.n_splits,
                                             a.max_blocks * kBlock, order);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kern<<<pl.n_splits * a.B * per, 32 * (warps + 1), smem, s>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

int attention_mma_row_tiles(const mtp_attn_args& a) {
  return (a.Hq / a.Hkv * (a.D + 1) + kGqaRowsPerCta - 1) / kGqaRowsPerCta;
}

bool attention_mma_supported(const mtp_attn_args& a) {
  if (a.dtype != MTP_BF16 || tensor_map_encoder() == nullptr) return false;
  if (a.is_mla) return a.d_qk == 576 && a.d_v == 512 && a.Hkv == 1;
  return a.d_qk == a.d_v && (a.d_qk == 64 || a.d_qk == 128);
}

cudaError_t launch_attention_mma(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  return a.d_qk == 128 ? run_gqa<128>(a, p, err, s) : run_gqa<64>(a, p, err, s);
}

bool attention_uses_mla_tc(const mtp_attn_args& a) { return a.is_mla && attention_mma_supported(a); }

cudaError_t launch_attention_mla(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s) {
  return launch_attention_mla_tc(a, p, err, s);
}

}  // namespace mtp
