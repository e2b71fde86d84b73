// GQA/MHA verify attention on the 5th-generation tensor cores, for KV heads
// that carry 49..64 query rows (group x R: e.g. 4 heads x 16 tree nodes, 8
// heads x 7 verify tokens), where the mma.sync kernel falls short of the
// cache read rate (up to 48 rows it reads the cache at 86-109 % of the
// measured copy rate).
//
// "Multi Token Prediction" note, K=3 flow step 2 (stacked queries against the
// reused cache, causal within the verify chain); tree drafts ("MTP in
// TensorRT-LLM on Blackwell", future work: tree speculative sampling, Fig. 9):
// each node sees the context and its root path. Row (j, g) = query head
// h*group+g of verify token j reads KV head h.
//
// Transposed formulation (keys on the TMEM lanes, rows on the columns):
//   S^T [128 keys x N rows]  = K_tile [128 x 128 dims] . Q^T      M = 128 keys
//   O^T [128 dv   x N rows] += V^T [128 dv x 128 keys] . P^T       M = 128 dv
// N = 64 (the KV head's rows, padding rows zero). TMEM: O^T in columns
// 0..63, two S^T buffers at 64 and 128.
//
// Shared memory: Q (two 64-dim chunks of [N rows x 128 B]) and three stages
// of one 128-key tile each: K slots (dims 0..63, 64..127) and V slots (dv
// 0..63, 64..127) of [128 keys x 64] (16 KB, 128-byte swizzle, keys 0..63
// from one cache block and 64..127 from the next). QK reads the K slots
// K-major, PV reads V^T MN-major from the two V slots, and P^T (bf16) goes
// into the tile's first K slot once QK is done. A stage is released after its
// PV, so the next tiles' loads stay in flight during the softmax. The MMA
// thread issues QK(g+1) as soon as tile g+1 has landed, so that it runs
// during the softmax of tile g, and PV(g) as soon as P(g) is written; P and
// the PV completions are signalled on barrier pairs indexed by g % 2, so no
// wait can mistake a phase two tiles old for the one it needs.
//
// Persistent CTAs, one per SM, each walking its share of the work items
// (split, request, KV head) in a longest-first order: the K/V producer runs on
// into the next item's tiles while the softmax warps finish the current one,
// so the stream from HBM does not stop at item boundaries.
//
// Warps: 0 MMA issuer, 1 K/V producer, 2 Q producer, 3 scheduler; 4..19
// softmax / epilogue: warp w owns TMEM lanes 32*(w%4)..+31 (keys of S^T, dv
// of O^T) and the 16 row columns 16*((w-4)/4)..+15.
//
// Online softmax with a lazy rescale (the reference row max only moves when a
// score exceeds it by more than 8 in log2 units; P and the row sums use the
// same reference, so the result is exact either way); each thread keeps
// partial row sums over its keys, reduced once after the last tile.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mtp {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box);

namespace {

constexpr int kKeys = 128;             // keys per tile (MMA M of S^T)
constexpr int kD = 128;                // head dim of K and V
constexpr int kTcMinRows = 49, kTcMaxRows = 64;   // query rows per KV head handled here
constexpr int kSlotBytes = 16384;      // [128 keys x 64 dims] bf16
constexpr int kStageBytes = 4 * kSlotBytes;   // K0, K1, V0, V1
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyRescale = 8.0f;   // log2 units

constexpr int kQOff = 0;                                   // 2 x [N rows x 128 B], at most 16 KB
constexpr int kStageOff = 16384;
constexpr int kRedOff = kStageOff + kStages * kStageBytes; // red_max[4][64], red_sum[4][64]
constexpr int kRowOff = kRedOff + 2 * 4 * 64 * 4;          // m_run, m_ref, rscale, path, m_shift [64]
constexpr int kRowOffOut = kRowOff + 5 * 64 * 4;           // int64 [64]: output element offset of each row
constexpr int kBarOff = kRowOffOut + 64 * 8;
constexpr int kRing = 8;                                   // work items published ahead by the scheduler warp
constexpr int kNumBars = 2 * kStages + 2 + 2 + 2 + 2 + 2 + 1 + 2 * kRing;
constexpr int kRingOff = kBarOff + kNumBars * 8;           // kRing work items (RingItem)
constexpr int kMiscOff = kRingOff + kRing * 32;            // TMEM base, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;

constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0;          // O^T: columns 0..N-1
constexpr uint32_t kColS = 64;         // S^T buffer b: 64 + 64 b

template <int kN>
struct Shape {
  static constexpr int kSoftWarps = kN / 4;              // 4 lane quarters x N/16 row quarters
  static constexpr int kSoftThreads = 32 * kSoftWarps;
  static constexpr int kThreads = 128 + kSoftThreads;
  static constexpr int kQChunk = kN * 128;               // one 64-dim chunk of Q; also one 64-key block of P^T
  static_assert(kN % 16 == 0 && kN <= 64, "row count");
};

struct Params {
  __nv_bfloat16* out;
  float* part_o;
  float* part_lse;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* order;    // work items, longest first (gqa_schedule_kernel)
  const int32_t* parents;  // [B, R] tree drafts, nullptr: chains
  unsigned* err;
  int B, R, Hq, Hkv, group, rows, max_blocks, num_blocks, split_len, n_splits;
  float scale_log2;
};

// A work item is (split, request, KV head): i = (split * B + b) * Hkv + h.
struct Item {
  int split, b, h;
};

__device__ __forceinline__ Item decode_item(int i, int B, int Hkv) {
  Item it;
  it.h = i % Hkv;
  it.b = (i / Hkv) % B;
  it.split = i / (Hkv * B);
  return it;
}

constexpr int kMaxItemTiles = 128;   // split_len <= 16384 keys

// Orders the work items by tile count, longest first (counting sort, one
// CTA) in groups of the Hkv items of one (split, request), which have the
// same keys: a request's KV heads share the cache blocks (the heads of a
// token are interleaved), so CTAs that start them together read the same
// DRAM pages at about the same time. CTAs take positions in index order, so
// long items start first and short ones fill the tail of the last round.
__global__ void __launch_bounds__(1024) gqa_schedule_kernel(const int32_t* __restrict__ ctx_lens, int B, int R,
                                                           int Hkv, int split_len, int n_splits, int max_len,
                                                           int32_t* __restrict__ order, unsigned* err) {
  __shared__ int hist[kMaxItemTiles + 1];
  const int n = n_splits * B;   // groups (split, request); group q = split * B + b holds items q * Hkv + h
  auto tiles_of = [&](int q) -> int {
    const int ctx = ctx_lens[q % B];
    if (ctx < 0 || ctx + R > max_len) {   // the attention kernel skips the request
      raise_error(err, MTP_ERR_LENGTH);
      return 0;
    }
    const int t0 = (q / B) * split_len;
    const int t_end = min(t0 + split_len, ctx + R);
    return t0 < t_end ? min((t_end - t0 + kKeys - 1) / kKeys, kMaxItemTiles) : 0;
  };
  for (int k = threadIdx.x; k <= kMaxItemTiles; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < n; q += blockDim.x) atomicAdd(&hist[tiles_of(q)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {   // hist[k] becomes the first group position of tile count k
    int acc = 0;
    for (int k = kMaxItemTiles; k >= 0; --k) {
      const int h = hist[k];
      hist[k] = acc;
      acc += h;
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const int pos = atomicAdd(&hist[tiles_of(q)], 1);
    for (int h = 0; h < Hkv; ++h) order[pos * Hkv + h] = q * Hkv + h;
  }
}

// MN-major operand with 128-byte swizzling: 64-element MN blocks `lbo` bytes
// apart, 8-row K groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(lbo >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

template <int kCount>
__device__ __forceinline__ void softmax_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCount) : "memory");
}

// Named barrier 1 over the softmax threads that also returns whether any of
// them passed true.
template <int kCount>
__device__ __forceinline__ bool softmax_barrier_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kCount)
      : "memory");
  return r != 0;
}

// 2^x with the hardware approximation (relative error ~2^-22, far below the
// bf16 rounding P goes through); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats to bf16 (round to nearest even): lo in bits 0..15, hi in 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void store_b16(uint8_t* p, uint32_t v) { *reinterpret_cast<uint16_t*>(p) = (uint16_t)v; }

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 values per lane: lane l (and l ^ 16) ends up with the op-reduction over
// all 32 lanes of element l % 16 (butterfly over lane bits 3..0, then one
// exchange across bit 4).
template <bool kMax>
__device__ __forceinline__ float transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = upper ? v[k] : v[k + w];
      const float keep = upper ? v[k + w] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float other = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], other) : v[0] + other;
}

// 32 lanes x 16 consecutive 32-bit columns (thread t: lane base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// The CTAs are persistent (one per SM): CTA c takes the items at positions
// r*G + c of the longest-first order in even rounds r and r*G + G-1-c in odd
// ones (G CTAs), so the long items spread over the SMs first and the short
// ones even out the loads. A scheduler warp walks that sequence (skipping
// items without keys) and publishes each item in a ring of kRing slots in
// shared memory, ahead of the roles that consume it, so that no role waits
// on the global loads an item takes at its start.
struct Cursor {
  int r = -1;   // round
  Item it;
  int ctx, t0, t_end, n_tiles;
};

__device__ __forceinline__ bool next_item(Cursor& c, const Params& p, int n_items) {
  const int G = gridDim.x, cta = blockIdx.x;
  while (true) {
    const int r = ++c.r;
    const int idx = r * G + ((r & 1) ? G - 1 - cta : cta);
    if (idx >= n_items) return false;
    c.it = decode_item(p.order[idx], p.B, p.Hkv);
    c.ctx = p.ctx_lens[c.it.b];
    if (c.ctx < 0 || c.ctx + p.R > p.max_blocks * kBlock) continue;   // reported by the schedule kernel
    c.t0 = c.it.split * p.split_len;
    c.t_end = min(c.t0 + p.split_len, c.ctx + p.R);
    if (c.t0 >= c.t_end) continue;   // no key of this split is visible: the combine skips it
    c.n_tiles = (c.t_end - c.t0 + kKeys - 1) / kKeys;
    return true;
  }
}

// One published work item; n_tiles == 0 ends the sequence.
struct RingItem {
  int b, h, split, ctx, t0, t_end, n_tiles, pad;
};

// Named barrier 1 over the softmax threads that also returns whether all of
// them passed true.
template <int kCount>
__device__ __forceinline__ bool softmax_barrier_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kCount)
      : "memory");
  return r != 0;
}

// kTree: rows see the verify keys of their root path (tree drafts); the chain
// instantiation keeps each row's plain key limit ctx + j in the same array.
template <int kN, bool kTree>
__global__ void __launch_bounds__(Shape<kN>::kThreads, 1) attn_gqa_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                           const __grid_constant__ CUtensorMap tm_k,
                                                                           const __grid_constant__ CUtensorMap tm_v,
                                                                           const Params p, const int n_items) {
  using S = Shape<kN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red_max = reinterpret_cast<float*>(smem + kRedOff);
  float* red_sum = red_max + 4 * 64;
  float* m_run = reinterpret_cast<float*>(smem + kRowOff);
  float* m_ref = m_run + 64;
  float* rscale = m_run + 128;
  uint32_t* path = reinterpret_cast<uint32_t*>(m_run + 192);   // per row: path mask (tree) or key limit (chain)
  float* m_shift = m_run + 256;
  int64_t* row_out = reinterpret_cast<int64_t*>(smem + kRowOffOut);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);   // [kStages]: the stage holds its tile
  uint64_t* empty = full + kStages;                                 // [kStages]: PV of the stage's tile is done
  uint64_t* qbar = empty + kStages;                                 // Q of the next item has landed
  uint64_t* q_empty = qbar + 1;                                     // the last QK of an item is done
  uint64_t* s_full = q_empty + 1;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;   // [2]: P of tile g published (barrier g % 2)
  uint64_t* o_done = p_full + 2;    // [2]: PV of tile g complete (barrier g % 2)
  uint64_t* final_bar = o_done + 2;
  uint64_t* item_full = final_bar + 1;   // [kRing]: the slot holds the next work item
  uint64_t* item_empty = item_full + kRing;   // [kRing]: every role has read the slot
  RingItem* ring = reinterpret_cast<RingItem*>(smem + kRingOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rows = p.rows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      sm100::mbar_init(&full[s], 1);
      sm100::mbar_init(&empty[s], 1);
    }
    sm100::mbar_init(qbar, 1);
    sm100::mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      sm100::mbar_init(&s_full[i], 1);
      sm100::mbar_init(&s_empty[i], S::kSoftWarps);
      sm100::mbar_init(&p_full[i], S::kSoftWarps);
      sm100::mbar_init(&o_done[i], 1);
    }
    sm100::mbar_init(final_bar, 1);
    for (int i = 0; i < kRing; ++i) {
      sm100::mbar_init(&item_full[i], 1);
      sm100::mbar_init(&item_empty[i], 3 + S::kSoftWarps);   // Q and K/V producers, MMA, softmax warps
    }
    *abort = 0;
    sm100::fence_barrier_init();
  }
  if (warp == 0) {
    sm100::tmem_alloc(tmem_slot, kTmemCols);
    sm100::tmem_relinquish();
  }
  // Padding rows of Q (rows .. kN-1 of both chunks) are zero: their scores
  // stay finite. The Q boxes only ever write rows 0 .. rows-1.
  for (int x = rows * 8 + (int)threadIdx.x; x < kN * 8; x += blockDim.x) {
    const int r = x / 8, c16 = x % 8;
#pragma unroll
    for (int c = 0; c < 2; ++c)
      *reinterpret_cast<uint4*>(smem + kQOff + c * S::kQChunk + r * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = sm100::smem_u32(smem);

  if (warp >= 4) {
    // ------------------------------------------------------- softmax warps
    const int sw = warp - 4;                 // 0 .. kSoftWarps-1
    const int qq = warp % 4;                 // TMEM lane quarter: keys / dv 32*qq + lane
    const int cq = sw >> 2;                  // row quarter: rows 16*cq .. 16*cq+15
    const int st = sw * 32 + lane;           // 0 .. kSoftThreads-1
    const uint32_t lane_addr = (uint32_t)(32 * qq) << 16;
    bool ok = true;
    int g = 0;                               // tiles of earlier items (stage, buffer and phase counter)
    for (int k = 0;; ++k) {
      // Every softmax thread has seen slot k published (and the previous
      // item's epilogue is done with the row state) before any goes on; a
      // failed wait anywhere stops them all together.
      const bool got = softmax_barrier_all<S::kSoftThreads>(
          ok && sm100::mbar_wait(&item_full[k % kRing], (uint32_t)((k / kRing) & 1), abort));
      if (!got) {
        ok = false;
        break;
      }
      const RingItem cur = ring[k % kRing];
      __syncwarp();
      if (lane == 0) sm100::mbar_arrive(&item_empty[k % kRing]);
      if (cur.n_tiles == 0) break;
      const int b = cur.b, h = cur.h, split = cur.split;
      const int ctx = cur.ctx, t0 = cur.t0, t_end = cur.t_end, n_tiles = cur.n_tiles;
      if (st < kN) {
        const int j = min(st, rows - 1) / p.group;   // padding rows copy the last row's mask
        path[st] = kTree ? tree_path_mask(p.parents, b, p.R, j, p.err) : (uint32_t)(ctx + j);
        m_run[st] = -INFINITY;
        m_ref[st] = 0.0f;
      }
      softmax_barrier<S::kSoftThreads>();
      float acc[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) acc[x] = 0.0f;
      // first key some row may not see: the first verify key of a tree, or
      // the key after row 0's own for a chain
      const int mask_from = kTree ? ctx : ctx + 1;
      for (int i = 0; i < n_tiles; ++i, ++g) {
        const int buf = g & 1;
        // S^T(g) is complete, and so is every MMA issued before QK(g): PV(g-2)
        // at least (QK(g) may have been issued before PV(g-1)).
        ok = ok && __all_sync(0xffffffffu, sm100::mbar_wait(&s_full[buf], (g >> 1) & 1, abort) ? 1 : 0);
        float d[16];   // score (log2 units) - reference max of the row
        if (ok) {
          sm100::tc_fence_after();
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem + lane_addr + kColS + buf * 64 + cq * 16, r);
          sm100::tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x) d[x] = fmaf(__uint_as_float(r[x]), p.scale_log2, -m_ref[cq * 16 + x]);
          sm100::tc_fence_before();
          __syncwarp();
          if (lane == 0) sm100::mbar_arrive(&s_empty[buf]);
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) d[x] = -INFINITY;
        }
        const int tile0 = t0 + i * kKeys;
        if (tile0 + kKeys - 1 >= mask_from || tile0 + kKeys > t_end) {   // causal / split edge inside the tile
          const int key = tile0 + 32 * qq + lane;
#pragma unroll
          for (int x = 0; x < 16; ++x)
            d[x] = (key >= t_end || (kTree ? tree_hidden(key, ctx, path[cq * 16 + x]) : key > (int)path[cq * 16 + x]))
                       ? -INFINITY
                       : d[x];
        }
        bool exceed = (i == 0);
#pragma unroll
        for (int x = 0; x < 16; ++x) exceed |= d[x] > kLazyRescale;
        if (softmax_barrier_any<S::kSoftThreads>(exceed)) {
          {
            float t[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) t[x] = d[x];
            const float mx = transpose_reduce16<true>(t, lane);   // max over the warp's 32 keys
            if (lane < 16) red_max[qq * 64 + cq * 16 + lane] = mx + m_ref[cq * 16 + lane];
          }
          softmax_barrier<S::kSoftThreads>();
          if (st < kN) {
            const float mt = fmaxf(fmaxf(red_max[st], red_max[64 + st]), fmaxf(red_max[128 + st], red_max[192 + st]));
            const float mo = m_run[st];
            float mn = mo, sc = 1.0f;
            if (mt > mo + kLazyRescale) {
              mn = mt;
              sc = (mo == -INFINITY) ? 0.0f : exp2f(mo - mn);
            }
            m_run[st] = mn;
            const float ref = mn == -INFINITY ? 0.0f : mn;   // rows with no visible key yet: p = 2^-inf = 0
            m_shift[st] = m_ref[st] - ref;
            m_ref[st] = ref;
            rscale[st] = sc;
          }
          softmax_barrier<S::kSoftThreads>();
          bool rescale = false;
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float sc = rscale[cq * 16 + x];
            rescale |= sc != 1.0f;
            acc[x] *= sc;
            d[x] += m_shift[cq * 16 + x];
          }
          // O^T columns of these rows hold PV up to tile g-1 once it completes
          // (QK(g) may have been issued before PV(g-1)): wait, then rescale.
          if (ok && i > 0 && __any_sync(0xffffffffu, rescale))
            ok = __all_sync(0xffffffffu,
                            sm100::mbar_wait(&o_done[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1), abort) ? 1 : 0);
          if (ok && i > 0 && rescale) {
            uint32_t r[16];
            const uint32_t ta = tmem + lane_addr + kColO + cq * 16;
            tmem_ld_32x32b_x16(ta, r);
            sm100::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * rscale[cq * 16 + x]);
            tmem_st_32x32b_x16(ta, r);
            tmem_st_wait();
          }
        }
        // p = 2^d: P^T (bf16) into the stage's first K slot as a K-major B
        // operand (block of 64 keys, row, key), and into the partial row sums.
        {
          const int k = 32 * qq + lane;
          uint8_t* pb = smem + kStageOff + (g % kStages) * kStageBytes + (k >> 6) * S::kQChunk;
          const int kin = k & 63;
#pragma unroll
          for (int x = 0; x < 16; x += 2) {   // rows r, r+1: one packed conversion, two 16-bit stores
            const float p0 = fast_exp2(d[x]), p1 = fast_exp2(d[x + 1]);
            acc[x] += p0;
            acc[x + 1] += p1;
            const int r = cq * 16 + x;
            const uint32_t pair = pack_bf16x2(p0, p1);
            store_b16(pb + r * 128 + ((((kin >> 3) ^ (r & 7))) << 4) + (kin & 7) * 2, pair);
            store_b16(pb + (r + 1) * 128 + ((((kin >> 3) ^ ((r + 1) & 7))) << 4) + (kin & 7) * 2, pair >> 16);
          }
        }
        fence_async_smem();
        sm100::tc_fence_before();
        __syncwarp();
        if (lane == 0 && ok) sm100::mbar_arrive(&p_full[g & 1]);
      }
      {   // row sums: over the warp's 32 keys, then over the 4 lane quarters
        const float sm = transpose_reduce16<false>(acc, lane);
        if (lane < 16) red_sum[qq * 64 + cq * 16 + lane] = sm;
      }
      softmax_barrier<S::kSoftThreads>();
      if (st < rows) {
        // Per row, once: 1/l (into rscale, free until the next item's first
        // tile), the offset of the row's output, and the split's log-sum-exp.
        const float l = red_sum[st] + red_sum[64 + st] + red_sum[128 + st] + red_sum[192 + st];
        rscale[st] = l > 0.0f ? 1.0f / l : 0.0f;
        const int j = st / p.group, gg = st - j * p.group;
        const int64_t orow = ((int64_t)b * p.R + j) * p.Hq + h * p.group + gg;
        row_out[st] = (p.n_splits == 1 ? orow : orow * p.n_splits + split) * kD;
        if (p.n_splits > 1 && ok)
          p.part_lse[orow * p.n_splits + split] = l > 0.0f ? (m_run[st] + log2f(l)) * kLn2 : -INFINITY;
      }
      // ------------------------------------------------------ epilogue
      // Wait for PV of the item's last tile (global tile g-1; with it every
      // earlier MMA). The next item's first PV waits for P, which these warps
      // publish only after reading O^T here.
      const bool done =
          ok && __all_sync(0xffffffffu, sm100::mbar_wait(&o_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort) ? 1 : 0);
      softmax_barrier<S::kSoftThreads>();
      if (done) {
        sm100::tc_fence_after();
        const int dv = 32 * qq + lane;
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem + lane_addr + kColO + cq * 16, r);
        sm100::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int rloc = cq * 16 + x;
          if (rloc >= rows) continue;
          const float o = __uint_as_float(r[x]) * rscale[rloc];
          const int64_t e = row_out[rloc] + dv;
          if (p.n_splits == 1) p.out[e] = __float2bfloat16_rn(o);
          else p.part_o[e] = o;
        }
        sm100::tc_fence_before();
      }
      // After a failed wait every softmax warp still walks the same items and
      // named barriers (no warp leaves the loop early), skipping the tensor
      // memory; the waits return at once once the abort flag is set.
    }
    if (!ok && lane == 0) {
      *abort = 1;
      raise_error(p.err, MTP_ERR_TIMEOUT);
    }
  } else if (warp >= 1 && warp <= 3 && lane == 0) {
    const uint64_t pol = sm100::l2_policy_evict_first();   // every cache byte is read by one CTA
    // Single-thread read of ring slot k: wait for it, copy it, release it.
    auto take = [&](int k, RingItem& out) -> bool {
      if (!sm100::mbar_wait(&item_full[k % kRing], (uint32_t)((k / kRing) & 1), abort)) return false;
      out = ring[k % kRing];
      sm100::mbar_arrive(&item_empty[k % kRing]);
      return true;
    };
    bool ok = true;
    if (warp == 3) {
      // ------------------------------------------------------- scheduler
      Cursor cur;
      for (int k = 0;; ++k) {
        const bool have = next_item(cur, p, n_items);
        const int s = k % kRing;
        ok = sm100::mbar_wait(&item_empty[s], (uint32_t)(((k / kRing) & 1) ^ 1), abort);
        if (!ok) break;
        RingItem r{};
        if (have) r = RingItem{cur.it.b, cur.it.h, cur.it.split, cur.ctx, cur.t0, cur.t_end, cur.n_tiles, 0};
        ring[s] = r;
        sm100::mbar_arrive(&item_full[s]);
        if (!have) break;
      }
    } else if (warp == 2) {
      // ------------------------------------------------------ Q producer
      // Q of item k (two boxes of [R tokens x group heads x 64 dims]) once
      // the last QK of item k-1 has read the previous one.
      sm100::tma_prefetch_desc(&tm_q);
      int k = 0;
      for (;; ++k) {
        RingItem it;
        ok = take(k, it);
        if (!ok || it.n_tiles == 0) break;
        ok = sm100::mbar_wait(q_empty, (uint32_t)((k & 1) ^ 1), abort);
        if (!ok) break;
        sm100::mbar_arrive_expect_tx(qbar, 2 * rows * 128);
        for (int c = 0; c < 2; ++c)
          sm100::tma_load_3d(smem + kQOff + c * S::kQChunk, &tm_q, qbar, c * 64, it.h * p.group, it.b * p.R, pol);
      }
      if (k > 0) sm100::mbar_wait_timeout(qbar, (uint32_t)((k - 1) & 1), sm100::kWaitTimeoutNs);
    } else {
      // ---------------------------------------------------- K/V producer
      // Per tile eight boxes of [64 keys x 64 dims]: K and V, dims 0..63
      // and 64..127, keys of the tile's two cache blocks; it runs on into
      // the next item's tiles while the current one is being finished. The
      // block ids of tile i+1 are read while tile i is issued. Keys past the
      // split end come from a block id of -1 (zero fill).
      sm100::tma_prefetch_desc(&tm_k);
      sm100::tma_prefetch_desc(&tm_v);
      constexpr int kNoBlock = INT_MIN;
      constexpr int kAhead = 4;   // L2 prefetch distance in tiles
      int g = 0;
      for (int k = 0; ok; ++k) {
        RingItem it;
        ok = take(k, it);
        if (!ok || it.n_tiles == 0) break;
        const int32_t* tbl = p.block_table + (int64_t)it.b * p.max_blocks;
        auto raw_block = [&](int key0) -> int { return key0 < it.t_end ? tbl[key0 / kBlock] : kNoBlock; };
        auto checked = [&](int v) -> int {   // cache block id, or -1 (zero fill)
          if (v == kNoBlock) return -1;
          if (v < 0 || v >= p.num_blocks) {
            raise_error(p.err, MTP_ERR_BLOCK_ID);
            return -1;
          }
          return v;
        };
        // Block ids of tiles i .. i+kAhead (two per tile), read kAhead+1
        // tiles ahead; tile i+kAhead is prefetched into L2 when tile i is
        // loaded, so its later load finds it there.
        int f0[kAhead + 1], f1[kAhead + 1];
#pragma unroll
        for (int j = 0; j <= kAhead; ++j) {
          f0[j] = raw_block(it.t0 + j * kKeys);
          f1[j] = raw_block(it.t0 + j * kKeys + 64);
        }
        auto prefetch = [&](int v) {   // the tile's boxes of one cache block (K and V, both dim halves)
          if (v == kNoBlock || v < 0 || v >= p.num_blocks) return;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            sm100::tma_prefetch_4d(&tm_k, c * 64, it.h, 0, v);
            sm100::tma_prefetch_4d(&tm_v, c * 64, it.h, 0, v);
          }
        };
        for (int i = 0; i < it.n_tiles; ++i, ++g) {
          const int b0 = f0[0], b1 = f1[0];
#pragma unroll
          for (int j = 0; j < kAhead; ++j) {
            f0[j] = f0[j + 1];
            f1[j] = f1[j + 1];
          }
          f0[kAhead] = raw_block(it.t0 + (i + kAhead + 1) * kKeys);
          f1[kAhead] = raw_block(it.t0 + (i + kAhead + 1) * kKeys + 64);
          const int s = g % kStages;
          ok = sm100::mbar_wait(&empty[s], (uint32_t)(((g / kStages) & 1) ^ 1), abort);
          if (!ok) break;
          sm100::mbar_arrive_expect_tx(&full[s], kStageBytes);
          uint8_t* stage = smem + kStageOff + s * kStageBytes;
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const int blk = checked(kb ? b1 : b0);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              sm100::tma_load_4d(stage + c * kSlotBytes + kb * 8192, &tm_k, &full[s], c * 64, it.h, 0, blk, pol);
              sm100::tma_load_4d(stage + (2 + c) * kSlotBytes + kb * 8192, &tm_v, &full[s], c * 64, it.h, 0, blk,
                                 pol);
            }
          }
          if (i == 0) {   // an item's first tiles: nothing prefetched them
#pragma unroll
            for (int j = 0; j + 1 < kAhead; ++j) {
              prefetch(f0[j]);
              prefetch(f1[j]);
            }
          }
          prefetch(f0[kAhead - 1]);   // tile i + kAhead
          prefetch(f1[kAhead - 1]);
        }
      }
      // Every copy must land before the CTA may exit: wait (time-limited)
      // for the last fill of each stage (g fills were issued).
      for (int s = 0; s < kStages && s < g; ++s) {
        const int last = s + (g - 1 - s) / kStages * kStages;
        sm100::mbar_wait_timeout(&full[s], (uint32_t)((last / kStages) & 1), sm100::kWaitTimeoutNs);
      }
    }
    if (!ok) {
      *abort = 1;
      raise_error(p.err, MTP_ERR_TIMEOUT);
    }
  } else if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- MMA
    // Tiles in order over all items (global tile g): QK(g) into S^T buffer
    // g%2, then (once P(g) is published) PV(g), whose completion releases
    // the stage to the producer and tells the epilogue. The first QK of an
    // item waits for its Q; the completion of its last QK frees Q for the
    // next item. The first PV of an item overwrites O^T.
    constexpr uint32_t idesc_qk = sm100::idesc_bf16_f32(128, kN);
    constexpr uint32_t idesc_pv = sm100::idesc_bf16_f32(128, kN) | (1u << 15);   // A (V^T) MN-major
    const uint64_t d_q = sm100::smem_desc_sw128_kmajor(smem_base + kQOff);
    // QK(g): S^T buffer g%2 from the stage's K slots. last: the tile is its
    // item's last (release Q once this QK is done).
    auto do_qk = [&](int g, bool last) {
      const int s = g % kStages, buf = g & 1;
      sm100::tc_fence_after();
      const uint32_t d = tmem + kColS + buf * 64;
      const uint64_t a0 = sm100::smem_desc_sw128_kmajor(smem_base + kStageOff + s * kStageBytes);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint64_t a = a0 + (uint64_t)(c * (kSlotBytes >> 4));
        const uint64_t q = d_q + (uint64_t)(c * (S::kQChunk >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) sm100::tc_mma_bf16(d, a + 2 * kk, q + 2 * kk, idesc_qk, (c | kk) ? 1u : 0u);
      }
      sm100::tc_commit(&s_full[buf]);
      if (last) sm100::tc_commit(q_empty);
    };
    // PV(g): O^T (+)= V^T P^T; its completion releases the stage and tells
    // the epilogue (and a rescale of O^T) that O^T holds tile g.
    auto do_pv = [&](int g, bool first) {
      const int s = g % kStages;
      sm100::tc_fence_after();
      const uint32_t sb = smem_base + kStageOff + s * kStageBytes;
      const uint64_t a0 = desc_mnmajor(sb + 2 * kSlotBytes, kSlotBytes);
      const uint64_t p0 = sm100::smem_desc_sw128_kmajor(sb);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        sm100::tc_mma_bf16(tmem + kColO, a0 + (uint64_t)(kk * (2048 >> 4)),
                           p0 + (uint64_t)(((kk >> 2) * S::kQChunk + (kk & 3) * 32) >> 4), idesc_pv,
                           (!first || kk > 0) ? 1u : 0u);
      sm100::tc_commit(&empty[s]);
      sm100::tc_commit(&o_done[g & 1]);
    };
    // Tile g may start once its S^T buffer is free, its keys have landed and
    // (first tile of an item: q_parity >= 0) its Q has.
    auto qk_ready = [&](int g, int q_parity) -> bool {
      return sm100::mbar_test_wait(&s_empty[g & 1], (uint32_t)(((g >> 1) & 1) ^ 1)) &&
             (q_parity < 0 || sm100::mbar_test_wait(qbar, (uint32_t)q_parity)) &&
             sm100::mbar_test_wait(&full[g % kStages], (uint32_t)((g / kStages) & 1));
    };
    // Issue PV(g) and, if there is a next tile, QK(g+1), each as soon as it
    // can start: QK(g+1) then runs during the softmax of tile g, and PV(g)
    // (which frees a stage) never waits for tile g+1's keys. Polls
    // without suspending; gives up after kWaitTimeoutNs or on abort.
    auto issue_step = [&](int g, bool first, bool next, int q_parity, bool next_last) -> bool {
      bool qk = !next, pv = false;
      const uint64_t start = sm100::globaltimer();
      uint32_t spins = 0;
      while (!(qk && pv)) {
        if (!qk && qk_ready(g + 1, q_parity)) {
          do_qk(g + 1, next_last);
          qk = true;
          continue;
        }
        if (!pv && sm100::mbar_test_wait(&p_full[g & 1], (uint32_t)((g >> 1) & 1))) {
          do_pv(g, first);
          pv = true;
          continue;
        }
        if (*abort) return false;
        if ((++spins & 255u) == 0 && sm100::globaltimer() - start > sm100::kWaitTimeoutNs) return false;
      }
      return true;
    };
    // Single-thread read of ring slot k: wait for it, copy it, release it.
    auto take = [&](int k, RingItem& out) -> bool {
      if (!sm100::mbar_wait(&item_full[k % kRing], (uint32_t)((k / kRing) & 1), abort)) return false;
      out = ring[k % kRing];
      sm100::mbar_arrive(&item_empty[k % kRing]);
      return true;
    };
    int g = 0, k = 0;
    RingItem cur;
    bool ok = take(0, cur);
    bool have = ok && cur.n_tiles > 0;
    if (have) {   // QK of the very first tile
      ok = sm100::mbar_wait(&s_empty[0], 1u, abort) && sm100::mbar_wait(qbar, 0u, abort) &&
           sm100::mbar_wait(&full[0], 0u, abort);
      if (ok) do_qk(0, cur.n_tiles == 1);
    }
    while (have && ok) {
      RingItem nxt;
      ok = take(k + 1, nxt);
      if (!ok) break;
      const bool have_next = nxt.n_tiles > 0;
      for (int i = 0; i < cur.n_tiles && ok; ++i, ++g) {
        const bool same = i + 1 < cur.n_tiles;   // the next tile belongs to this item
        ok = issue_step(g, i == 0, same || have_next, same ? -1 : ((k + 1) & 1),
                        same ? i + 2 == cur.n_tiles : nxt.n_tiles == 1);
      }
      cur = nxt;
      have = have_next;
      ++k;
    }
    if (!ok) {
      *abort = 1;
      raise_error(p.err, MTP_ERR_TIMEOUT);
    }
    sm100::tc_commit(final_bar);
    sm100::mbar_wait_timeout(final_bar, 0, sm100::kWaitTimeoutNs);
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem, kTmemCols);
  }
}

using GqaTcKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const Params, const int);

template <int kN>
GqaTcKernel pick(bool tree) {
  return tree ? attn_gqa_tc_kernel<kN, true> : attn_gqa_tc_kernel<kN, false>;
}

template <int kN>
cudaError_t launch_n(bool tree, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const Params& p,
                     int n_items, int sm_count, cudaStream_t s) {
  const GqaTcKernel kern = pick<kN>(tree);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(n_items, sm_count));   // persistent: one CTA per SM
  kern<<<grid, Shape<kN>::kThreads, kSmemBytes, s>>>(tq, tk, tv, p, n_items);
  return cudaGetLastError();
}

}  // namespace

bool attention_uses_gqa_tc(const mtp_attn_args& a) {
  if (a.is_mla || a.dtype != MTP_BF16 || a.d_qk != kD || a.d_v != kD) return false;
  if (a.Hkv <= 0 || a.Hq % a.Hkv != 0 || tensor_map_encoder() == nullptr) return false;
  const int rows = (a.Hq / a.Hkv) * (a.D + 1);
  return rows >= kTcMinRows && rows <= kTcMaxRows;
}

int gqa_tc_split_granularity() { return kKeys; }

cudaError_t launch_attention_gqa_tc(const mtp_attn_args& a, const AttnPlan& pl, unsigned* err, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  const int R = a.D + 1, group = a.Hq / a.Hkv, rows = group * R;
  if (pl.split_len % kKeys || rows > kTcMaxRows || rows < kTcMinRows) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.Hq, (cuuint64_t)a.B * R};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a.Hq * kD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)R};
    if (!make_bf16_map(&tq, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)a.Hkv, (cuuint64_t)kBlock, (cuuint64_t)a.num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)a.Hkv * kD * 2,
                                   (cuuint64_t)kBlock * a.Hkv * kD * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kBlock, 1};
    if (!make_bf16_map(&tk, a.k_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_bf16_map(&tv, a.v_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  Params p;
  p.out = (__nv_bfloat16*)a.out;
  p.part_o = pl.n_splits > 1 ? (float*)((char*)a.workspace + pl.ws_partial_o) : nullptr;
  p.part_lse = pl.n_splits > 1 ? (float*)((char*)a.workspace + pl.ws_partial_lse) : nullptr;
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.order = (const int32_t*)((const char*)a.workspace + pl.ws_order);
  p.parents = a.parents;
  p.err = err;
  p.B = a.B;
  p.R = R;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = group;
  p.rows = rows;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.scale_log2 = a.sm_scale * kLog2e;
  const int n_items = pl.n_splits * a.B * a.Hkv;
  gqa_schedule_kernel<<<1, 1024, 0, s>>>(a.ctx_lens, a.B, R, a.Hkv, pl.split_len, pl.n_splits, a.max_blocks * kBlock,
                                         (int32_t*)((char*)a.workspace + pl.ws_order), err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const bool tree = a.parents != nullptr;
  return launch_n<64>(tree, tq, tk, tv, p, n_items, std::max(1, pl.sm_count), s);
}

}  // namespace mtp
