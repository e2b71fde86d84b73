// LM head on the 5th-generation tensor cores (tcgen05 MMA into TMEM, TMA
// loads, mbarrier pipeline) with the softmax statistics fused into the
// epilogue, for bf16 weights.
//
// "Multi Token Prediction" note, K=3 flow step 4: Logits_i = H_i x W_o for
// all verify rows in one product; step 5: softmax over the vocabulary. The
// full logits are never stored for greedy rows: the epilogue keeps, per row,
// a running max, sum of exp(l - max) and argmax over the vocabulary this CTA
// sees; rejection-sampling rows also get their fp32 logit rows written once
// (their residual draw needs the whole row after the log-sum-exp is known),
// and relaxed rows count the entries that rank before their draft ("MTP in
// TensorRT-LLM on Blackwell", relaxed acceptance; relaxed_count).
//
// Mapping (swap-AB): the MMA's M dimension is 128 vocabulary rows of W (the
// big streamed operand), its N dimension is a group of N verify rows of
// hidden (N = 32..256), K runs over the hidden size in 64-element steps, so
// one accumulator tile is 128 (vocab, TMEM lanes) x N (rows, TMEM columns)
// fp32. Persistent CTAs: row group g of the hidden rows is served by
// `cpg` CTAs that walk the vocabulary tiles t = s, s + cpg, ...
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM
// and issues the MMAs, warps 2..5 are the epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31). Two TMEM accumulators let the epilogue of tile i overlap
// the MMAs of tile i+1.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mtp {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box);

namespace {

constexpr int kThreadsTc = 192;
constexpr int kTileV = 128;          // vocab rows per MMA tile (MMA M)
constexpr int kTileK = 64;           // hidden elements per pipeline stage (128 B rows, 128-B swizzle)
constexpr int kMaxN = 256;           // rows per row group (MMA N)
constexpr int kSmemLimit = 232448;   // 227 KB opt-in per CTA
constexpr int kMaxStages = 8;

struct TcParams {
  const int32_t* tokens;
  const uint8_t* mode;
  const float* temperature;
  float* pmax;
  float* psum;
  float* pbest;
  int* pidx;
  float* ldraft;
  float* samp_logits;   // [M, V], rows of sampling requests only (nullptr: none)
  float* logits_debug;  // [M, V] optional
  const float* lpre;    // [M] draft logits of relaxed rows (NaN: not relaxed), nullptr: no relaxed request
  int* rcnt;            // [3][cpg][M] relaxed rank counts per CTA
  unsigned* err;
  int any_sampling;
  int M, R, H, V;
  int N;                // rows per group (multiple of 32)
  int cpg;              // CTAs per row group
  int n_tiles;          // vocab tiles
  int stages;
  uint32_t tmem_cols;   // allocated TMEM columns (power of 2 >= 2N); accumulator b at b * tmem_cols / 2
};

struct SmemLayout {
  int a_off, b_off, stage_bytes, bar_off, misc_off, epi_off, rows_off, total;
};

// pair: the CTA holds half of the group's N rows of hidden (CTA-pair MMA).
__host__ __device__ inline SmemLayout smem_layout(int N, int stages, bool pair) {
  SmemLayout L;
  const int a_bytes = kTileV * kTileK * 2;       // 16 KB
  const int b_bytes = (pair ? N / 2 : N) * kTileK * 2;   // rows x 128 B
  L.stage_bytes = a_bytes + b_bytes;
  L.a_off = 0;                                   // stage s: A at s*stage_bytes, B right after A
  L.b_off = a_bytes;
  int off = stages * L.stage_bytes;              // multiple of 1024 (a_bytes and b_bytes are)
  L.bar_off = off;
  off += (2 * stages + 5) * 8;                   // full[], empty[], acc_full[2], acc_empty[2], final
  L.misc_off = off;
  off += 16;                                     // TMEM base, abort flag
  off = (off + 15) / 16 * 16;
  L.epi_off = off;
  off += 4 * 32 * 33 * 4;                        // per-epilogue-warp 32x33 transpose buffers (later: 4 x N row stats)
  L.rows_off = off;
  off += N * 28;                                 // per-row draft id, 1/T, sampling flag, relaxed draft logit, 3 counts
  L.total = off + 1024;                          // + alignment slack for the 1024-B aligned base
  return L;
}

__device__ __forceinline__ void abort_all(volatile int* abort, unsigned* err) {
  *abort = 1;
  raise_error(err, MTP_ERR_TIMEOUT);
}

// kPair: CTA pairs (clusters of 2) share each MMA: a pair covers 256 vocab
// rows per tile (128 per CTA, its A half) and each CTA stages half of the
// group's hidden rows (its B half), so each SM streams half of the hidden
// tile through shared memory. The even CTA issues the MMAs; both CTAs' loads
// of a stage complete on the even CTA's full barrier.
template <int NCH, bool kPair>
__global__ void __launch_bounds__(kThreadsTc, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                     const TcParams p) {
  constexpr int N = NCH * 32;
  constexpr int kBRows = kPair ? N / 2 : N;      // hidden rows staged by this CTA
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout L = smem_layout(N, p.stages, kPair);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* final_bar = acc_empty + 2;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
  float* epi_buf = reinterpret_cast<float*>(smem + L.epi_off);
  int* row_draft = reinterpret_cast<int*>(smem + L.rows_off);
  float* row_inv_t = reinterpret_cast<float*>(smem + L.rows_off + N * 4);
  int* row_samp = reinterpret_cast<int*>(smem + L.rows_off + N * 8);
  float* row_lpre = reinterpret_cast<float*>(smem + L.rows_off + N * 12);
  int* row_cnt = reinterpret_cast<int*>(smem + L.rows_off + N * 16);   // [N][3]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int group = blockIdx.x / p.cpg;
  const int cta_in_group = blockIdx.x % p.cpg;   // also the partial-statistics slice of this CTA
  const int row0 = group * N;
  const int k_steps = p.H / kTileK;
  const uint32_t rank = kPair ? sm100::cluster_ctarank() : 0u;   // == cta_in_group % 2 (cpg is even)
  const bool leader = rank == 0;
  // Vocabulary units: 128 rows (one CTA) or 256 rows (a pair, 128 per CTA).
  constexpr int kUnit = kPair ? 2 * kTileV : kTileV;
  const int slot = kPair ? cta_in_group / 2 : cta_in_group;
  const int nslots = kPair ? p.cpg / 2 : p.cpg;
  const int n_units = (p.V + kUnit - 1) / kUnit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      sm100::mbar_init(&full[s], 1);
      sm100::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      sm100::mbar_init(&acc_full[b], 1);
      sm100::mbar_init(&acc_empty[b], kPair ? 8 : 4);   // epilogue warps of both CTAs drain it
    }
    sm100::mbar_init(final_bar, 1);
    *abort = 0;
    sm100::fence_barrier_init();
    sm100::tma_prefetch_desc(&tm_w);
    sm100::tma_prefetch_desc(&tm_h);
  }
  if (warp == 1) {
    if (kPair) {
      sm100::tmem_alloc_pair(tmem_base_slot, p.tmem_cols);
      sm100::tmem_relinquish_pair();
    } else {
      sm100::tmem_alloc(tmem_base_slot, p.tmem_cols);
      sm100::tmem_relinquish();
    }
  }
  // Per-row information of this CTA's row group.
  for (int r = threadIdx.x; r < N; r += kThreadsTc) {
    const int m = row0 + r;
    int draft = -1, samp = 0;
    float inv_t = 1.0f;
    if (m < p.M) {
      const int b = m / p.R, j = m % p.R;
      if (p.any_sampling && p.mode[b] == 1 && p.temperature[b] > 0.0f) {
        samp = 1;
        inv_t = 1.0f / p.temperature[b];
      }
      if (j < p.R - 1) draft = p.tokens[m + 1];
    }
    row_draft[r] = draft;
    row_inv_t[r] = inv_t;
    row_samp[r] = samp;
    row_lpre[r] = (p.lpre && m < p.M) ? p.lpre[m] : __int_as_float(0x7fc00000);
    row_cnt[3 * r] = row_cnt[3 * r + 1] = row_cnt[3 * r + 2] = 0;
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (kPair) sm100::cluster_sync();   // the peer's barriers and TMEM exist before any remote arrive or MMA
  sm100::tc_fence_after();
  const uint32_t tmem_base = *tmem_base_slot;

  // Units of this CTA (pair): u = slot + i * nslots; its vocabulary rows
  // start at u * kUnit + rank * 128.
  const int my_tiles = slot < n_units ? (n_units - 1 - slot) / nslots + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = sm100::l2_policy_evict_first();
      const uint64_t pol_h = sm100::l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int v0 = (slot + i * nslots) * kUnit + (int)rank * kTileV;
        for (int k = 0; k < k_steps; ++k) {
          const bool free_ = kPair ? sm100::mbar_wait_cluster(&empty[stage], phase ^ 1u, abort)
                                   : sm100::mbar_wait(&empty[stage], phase ^ 1u, abort);
          if (!free_) {
            abort_all(abort, p.err);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * L.stage_bytes;
          if (kPair) {
            // both CTAs' halves complete on the leader's full barrier
            if (leader) sm100::mbar_arrive_expect_tx(&full[stage], 2 * L.stage_bytes);
            sm100::tma_load_2d_pair(st + L.a_off, &tm_w, &full[stage], 0, k * kTileK, v0, pol_w);
            sm100::tma_load_2d_pair(st + L.b_off, &tm_h, &full[stage], 0, k * kTileK, row0 + (int)rank * kBRows,
                                    pol_h);
          } else {
            sm100::mbar_arrive_expect_tx(&full[stage], L.stage_bytes);
            sm100::tma_load_2d(st + L.a_off, &tm_w, &full[stage], k * kTileK, v0, pol_w);
            sm100::tma_load_2d(st + L.b_off, &tm_h, &full[stage], k * kTileK, row0, pol_h);
          }
          ++issued;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every issued load must have landed before the CTA exits: wait (time
      // limited) for the completion of the most recent fill of each stage.
      // (A pair's loads all complete on the leader's barriers; the odd CTA
      // leaves only after the closing cluster barrier.)
      for (int j = 0; j < (kPair && !leader ? 0 : min(issued, p.stages)); ++j) {
        const int idx = issued - 1 - j;
        sm100::mbar_wait_timeout(&full[idx % p.stages], (uint32_t)((idx / p.stages) & 1), sm100::kWaitTimeoutNs);
      }
    }
  } else if (warp == 1 && (!kPair || leader)) {
    // ---------------------------------------------------------- MMA issue
    // The whole warp runs the loop (descriptors stay warp-uniform) and one
    // elected lane issues. Two pipeline stages are waited for together and
    // their eight MMAs go out back to back: every wait or tcgen05 fence in
    // the issue stream costs the warp a few hundred clocks (measured), about
    // the time of one stage's MMAs.
    constexpr uint32_t idesc = sm100::idesc_bf16_f32(kPair ? 2 * kTileV : kTileV, N);
    auto landed = [&](int st, uint32_t ph) -> bool {
      const bool r = kPair ? sm100::mbar_poll_cluster(&full[st], ph, abort) : sm100::mbar_wait(&full[st], ph, abort);
      return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < my_tiles && ok; ++i) {
      const int buf = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      const bool drained = kPair ? sm100::mbar_poll_cluster(&acc_empty[buf], acc_phase ^ 1u, abort)
                                 : sm100::mbar_wait(&acc_empty[buf], acc_phase ^ 1u, abort);
      if (!__all_sync(0xffffffffu, drained ? 1 : 0)) {
        if (lane == 0) abort_all(abort, p.err);
        break;
      }
      sm100::tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * (p.tmem_cols / 2);
      for (int k = 0; k < k_steps;) {
        const int nk = k + 1 < k_steps ? 2 : 1;
        int st2 = stage + 1;
        uint32_t ph2 = phase;
        if (st2 == p.stages) {
          st2 = 0;
          ph2 ^= 1u;
        }
        if (!landed(stage, phase) || (nk == 2 && !landed(st2, ph2))) {
          if (lane == 0) abort_all(abort, p.err);
          ok = false;
          break;
        }
        sm100::tc_fence_after();
        if (sm100::elect_one()) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u < nk) {
              const int su = u == 0 ? stage : st2;
              const uint64_t adesc = sm100::smem_desc_sw128_kmajor(sm100::smem_u32(smem + su * L.stage_bytes + L.a_off));
              const uint64_t bdesc = sm100::smem_desc_sw128_kmajor(sm100::smem_u32(smem + su * L.stage_bytes + L.b_off));
#pragma unroll
              for (int kk = 0; kk < kTileK / 16; ++kk) {
                // Advance 16 elements (32 B) along K inside the 128-B swizzled row.
                const uint32_t acc = (k + u > 0 || kk > 0) ? 1u : 0u;
                if (kPair)
                  sm100::tc_mma_bf16_pair(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, acc);
                else
                  sm100::tc_mma_bf16(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, acc);
              }
              // stage free (in both CTAs of a pair) once these MMAs have read it
              if (kPair) sm100::tc_commit_pair_mc(&empty[su], 3);
              else sm100::tc_commit(&empty[su]);
            }
          }
        }
        __syncwarp();
        for (int u = 0; u < nk; ++u)
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        k += nk;
      }
      if (ok) {
        if (sm100::elect_one()) {
          if (kPair) sm100::tc_commit_pair_mc(&acc_full[buf], 3);
          else sm100::tc_commit(&acc_full[buf]);
        }
        __syncwarp();
      }
    }
    // Every MMA issued so far has completed before TMEM is released.
    if (sm100::elect_one()) {
      if (kPair) sm100::tc_commit_pair_mc(final_bar, 3);
      else sm100::tc_commit(final_bar);
    }
    __syncwarp();
    sm100::mbar_wait_timeout(final_bar, 0, sm100::kWaitTimeoutNs);
  } else if (warp == 1) {
    // pair, odd CTA: the even CTA's MMAs write this CTA's TMEM; wait for the
    // last one before the closing barriers.
    if (lane == 0) sm100::mbar_wait_timeout(final_bar, 0, sm100::kWaitTimeoutNs);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp % 4;                       // TMEM lane quarter
    float* tb = epi_buf + (warp - 2) * 32 * 33;   // this warp's transpose buffer
    RowStat st[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) st[c] = rowstat_empty();
    for (int i = 0; i < my_tiles; ++i) {
      const int buf = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      const bool ok = __all_sync(0xffffffffu, (kPair ? sm100::mbar_wait_cluster(&acc_full[buf], acc_phase, abort)
                                                     : sm100::mbar_wait(&acc_full[buf], acc_phase, abort))
                                                  ? 1
                                                  : 0) != 0;
      if (!ok) {
        if (lane == 0) abort_all(abort, p.err);
        break;
      }
      sm100::tc_fence_after();
      const int vbase = (slot + i * nslots) * kUnit + (int)rank * kTileV + 32 * q;   // vocab of lane 0 of this warp
      const int nvalid = min(32, p.V - vbase);                          // may be <= 0 in the tail tile
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        uint32_t r[32];
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + buf * (p.tmem_cols / 2) + c * 32;
        sm100::tmem_ld_32x32b_x32(taddr, r);
        sm100::tmem_ld_wait();
        // r[x] = logit(vocab vbase + lane, row c*32 + x): transpose so that
        // this thread then owns row c*32 + lane across the warp's 32 vocab.
#pragma unroll
        for (int x = 0; x < 32; ++x) tb[x * 33 + lane] = __uint_as_float(r[x]);
        __syncwarp();
        const int rr = c * 32 + lane;
        const int m = row0 + rr;
        if (m < p.M && nvalid > 0) {
          const bool samp = row_samp[rr] != 0;
          const float inv_t = row_inv_t[rr];
          float* rowv = tb + lane * 33;
          float cmax = -INFINITY;
          int cidx = 0;
          for (int x = 0; x < nvalid; ++x) {
            float l = rowv[x];
            if (samp) l = __fmul_rn(l, inv_t);
            rowv[x] = l;
            if (l > cmax) {
              cmax = l;
              cidx = x;
            }
          }
          float csum = 0.0f;
          for (int x = 0; x < nvalid; ++x) csum += expf(rowv[x] - cmax);
          st[c] = rowstat_merge(st[c], RowStat{cmax, csum, cmax, vbase + cidx});
          const int d = row_draft[rr];
          if (d >= vbase && d < vbase + nvalid) p.ldraft[m] = rowv[d - vbase];
          const float lp = row_lpre[rr];
          if (lp == lp) {   // relaxed row: rank counts of its draft over these entries
            const float eps = kRelaxedRankEps * (1.0f + fabsf(lp));
            int c0 = 0, c1 = 0, c2 = 0;
            for (int x = 0; x < nvalid; ++x) relaxed_count(rowv[x], vbase + x, lp, d, eps, c0, c1, c2);
            atomicAdd(&row_cnt[3 * rr], c0);
            atomicAdd(&row_cnt[3 * rr + 1], c1);
            atomicAdd(&row_cnt[3 * rr + 2], c2);
          }
          if (!(nvalid == 32 && (p.V & 3) == 0)) {   // ragged vocabulary tail: this lane writes its row
            float* dst_s = (samp && p.samp_logits) ? p.samp_logits + (int64_t)m * p.V + vbase : nullptr;
            float* dst_d = p.logits_debug ? p.logits_debug + (int64_t)m * p.V + vbase : nullptr;
            for (int x = 0; x < nvalid; ++x) {
              if (dst_s) dst_s[x] = rowv[x];
              if (dst_d) dst_d[x] = rowv[x];
            }
          }
        }
        // Whole 32-entry slices: the warp writes the chunk's rows from the
        // transpose buffer, eight lanes per row, so every store instruction
        // fills four whole 128-byte lines (a lane writing its own row would
        // touch 32 lines per instruction, and that L1 traffic competes with
        // the MMAs' operand reads for the same shared-memory bandwidth).
        if (nvalid == 32 && (p.V & 3) == 0 &&
            __any_sync(0xffffffffu, row0 + c * 32 + lane < p.M && (p.logits_debug || (p.samp_logits && row_samp[c * 32 + lane])))) {
          __syncwarp();
          const int x0 = 4 * (lane & 7);
#pragma unroll 1
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const int m2 = row0 + c * 32 + r;
            if (m2 < p.M) {
              const float* src = tb + r * 33 + x0;
              const float4 v4 = make_float4(src[0], src[1], src[2], src[3]);
              const int64_t o = (int64_t)m2 * p.V + vbase + x0;
              // streaming stores: the rows are read once, later, by the race
              // kernel; W tiles shared by the row groups stay in L2
              if (p.samp_logits && row_samp[c * 32 + r]) __stcs(reinterpret_cast<float4*>(p.samp_logits + o), v4);
              if (p.logits_debug) *reinterpret_cast<float4*>(p.logits_debug + o) = v4;
            }
          }
        }
        __syncwarp();
      }
      sm100::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair) sm100::mbar_arrive_remote_relaxed(&acc_empty[buf], 0);   // TMEM reads done: nothing to publish
        else sm100::mbar_arrive(&acc_empty[buf]);
      }
    }
    // Merge the four lane quarters' statistics through shared memory, then
    // write one partial per (CTA, row): slice = cta_in_group.
    asm volatile("bar.sync 1, 128;" ::: "memory");            // every epilogue warp is done with its buffer
    RowStat* ex = reinterpret_cast<RowStat*>(epi_buf);         // [4][N]
#pragma unroll
    for (int c = 0; c < NCH; ++c) ex[q * N + c * 32 + lane] = st[c];
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int r = (warp - 2) * 32 + lane; r < N; r += 128) {
      const int m = row0 + r;
      if (m >= p.M) continue;
      RowStat a = rowstat_merge(rowstat_merge(ex[r], ex[N + r]), rowstat_merge(ex[2 * N + r], ex[3 * N + r]));
      const int64_t o = (int64_t)cta_in_group * p.M + m;
      p.pmax[o] = a.m;
      p.psum[o] = a.s;
      p.pbest[o] = a.best;
      p.pidx[o] = a.idx;
      if (p.rcnt) {
        const int64_t plane = (int64_t)p.cpg * p.M;
        p.rcnt[o] = row_cnt[3 * r];
        p.rcnt[plane + o] = row_cnt[3 * r + 1];
        p.rcnt[2 * plane + o] = row_cnt[3 * r + 2];
      }
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (kPair) sm100::cluster_sync();   // both CTAs done with TMEM and with each other's barriers
  if (warp == 1) {
    sm100::tc_fence_after();
    if (kPair) sm100::tmem_dealloc_pair(tmem_base, p.tmem_cols);
    else sm100::tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ------------------------------------------------------------------- host
// 2D bf16 row-major [rows, cols] tensor, box {64 columns, box_rows rows},
// 128-byte swizzle, out-of-bounds rows read as zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, box_rows};
  return make_bf16_map(map, base, 2, dims, strides, box);
}

struct TcShape {
  int N, groups, cpg, stages;
  bool pair;
  uint32_t tmem_cols;
};

// CTA pairs from 33 verify rows on: a pair halves the hidden tile that each
// SM restages for every vocabulary tile, which relieves shared memory even
// where W's stream sets the pace (measured on the GB300: 64..192 rows 1-3 %
// faster, 32 rows unchanged). Fewer rows keep single-CTA tiles.
constexpr int kPairMinRows = 33;

template <int NCH, bool kPair>
cudaError_t set_smem(int smem) {
  return cudaFuncSetAttribute(lmhead_tc_kernel<NCH, kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// How many 2-CTA clusters of the pair kernel for this N can be resident at
// once (the persistent grid must not exceed it, or a second wave would run).
template <int NCH>
int pair_clusters(int stages) {
  const int smem = smem_layout(NCH * 32, stages, true).total;
  if (set_smem<NCH, true>(smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreadsTc, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, lmhead_tc_kernel<NCH, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int pair_clusters_for(int nch, int stages) {
  switch (nch) {
    case 1: return pair_clusters<1>(stages);
    case 2: return pair_clusters<2>(stages);
    case 3: return pair_clusters<3>(stages);
    case 4: return pair_clusters<4>(stages);
    case 5: return pair_clusters<5>(stages);
    case 6: return pair_clusters<6>(stages);
    case 7: return pair_clusters<7>(stages);
    case 8: return pair_clusters<8>(stages);
    default: return 0;
  }
}

// Resident 2-CTA clusters per (device, N), queried once.
int cached_pair_clusters(int nch, int stages) {
  static std::mutex mu;
  static int cache[64][9];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& row : cache)
      for (int& v : row) v = -1;
    init = true;
  }
  if (cache[dev][nch] < 0) cache[dev][nch] = pair_clusters_for(nch, stages);
  return cache[dev][nch];
}

TcShape tc_shape(int M, int sm_count) {
  TcShape s;
  s.groups = (M + kMaxN - 1) / kMaxN;
  const int per = (M + s.groups - 1) / s.groups;
  s.N = std::max(32, (per + 31) / 32 * 32);
  s.pair = M >= kPairMinRows;
  s.stages = kMaxStages;
  while (s.stages > 2 && smem_layout(s.N, s.stages, s.pair).total > kSmemLimit) --s.stages;
  s.cpg = std::max(1, sm_count / s.groups);
  if (s.pair) {
    const int clusters = std::min(sm_count / 2, cached_pair_clusters(s.N / 32, s.stages));
    if (clusters >= s.groups) s.cpg = 2 * (clusters / s.groups);
    else s.pair = false;   // cannot place one pair per group: single-CTA tiles
    if (!s.pair) {
      s.stages = kMaxStages;
      while (s.stages > 2 && smem_layout(s.N, s.stages, false).total > kSmemLimit) --s.stages;
    }
  }
  s.tmem_cols = 64;
  while (s.tmem_cols < (uint32_t)(2 * s.N)) s.tmem_cols *= 2;
  return s;
}

template <int NCH>
cudaError_t launch_nch(const TcShape& sh, const CUtensorMap& tw, const CUtensorMap& th, const TcParams& p,
                       cudaStream_t s) {
  const int smem = smem_layout(NCH * 32, sh.stages, sh.pair).total;
  if (!sh.pair) {
    cudaError_t e = set_smem<NCH, false>(smem);
    if (e != cudaSuccess) return e;
    lmhead_tc_kernel<NCH, false><<<sh.groups * sh.cpg, kThreadsTc, smem, s>>>(tw, th, p);
    return cudaGetLastError();
  }
  cudaError_t e = set_smem<NCH, true>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.groups * sh.cpg, 1, 1);
  cfg.blockDim = dim3(kThreadsTc, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, lmhead_tc_kernel<NCH, true>, tw, th, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool lmhead_tc_supported(const mtp_lmhead_args& a) {
  return a.dtype == MTP_BF16 && a.H % kTileK == 0 && tensor_map_encoder() != nullptr;
}

int lmhead_tc_slices(int V, int M, int sm_count) {
  (void)V;
  return tc_shape(M, sm_count).cpg;
}

cudaError_t launch_lmhead_tc(const mtp_lmhead_args& a, const LmPlan& pl, unsigned* err, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const TcShape sh = tc_shape(pl.M, sms);
  if (sh.cpg != pl.slices) return cudaErrorInvalidValue;
  CUtensorMap tw, th;
  if (!make_map(&tw, a.lm_head, (uint64_t)a.V, (uint64_t)a.H, kTileV)) return cudaErrorInvalidValue;
  if (!make_map(&th, a.hidden, (uint64_t)pl.M, (uint64_t)a.H, (uint32_t)(sh.pair ? sh.N / 2 : sh.N)))
    return cudaErrorInvalidValue;
  char* ws = (char*)a.workspace;
  TcParams p;
  p.tokens = a.tokens;
  p.mode = a.mode;
  p.temperature = a.temperature;
  p.pmax = (float*)(ws + pl.off_pmax);
  p.psum = (float*)(ws + pl.off_psum);
  p.pbest = (float*)(ws + pl.off_pbest);
  p.pidx = (int*)(ws + pl.off_pidx);
  p.ldraft = (float*)(ws + pl.off_ldraft);
  p.samp_logits = a.any_sampling ? (float*)(ws + pl.off_logits) : nullptr;
  p.logits_debug = a.logits_debug;
  p.lpre = a.relaxed_topk > 0 ? (const float*)(ws + pl.off_lpre) : nullptr;
  p.rcnt = a.relaxed_topk > 0 ? (int*)(ws + pl.off_rcnt) : nullptr;
  p.err = err;
  p.any_sampling = a.any_sampling;
  p.M = pl.M;
  p.R = a.D + 1;
  p.H = a.H;
  p.V = a.V;
  p.N = sh.N;
  p.cpg = sh.cpg;
  p.n_tiles = (a.V + kTileV - 1) / kTileV;
  p.stages = sh.stages;
  p.tmem_cols = sh.tmem_cols;
  switch (sh.N / 32) {
    case 1: return launch_nch<1>(sh, tw, th, p, s);
    case 2: return launch_nch<2>(sh, tw, th, p, s);
    case 3: return launch_nch<3>(sh, tw, th, p, s);
    case 4: return launch_nch<4>(sh, tw, th, p, s);
    case 5: return launch_nch<5>(sh, tw, th, p, s);
    case 6: return launch_nch<6>(sh, tw, th, p, s);
    case 7: return launch_nch<7>(sh, tw, th, p, s);
    case 8: return launch_nch<8>(sh, tw, th, p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mtp
