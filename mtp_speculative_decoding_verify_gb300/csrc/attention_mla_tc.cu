// Absorbed-MLA verify attention on the 5th-generation tensor cores.
//
// "Multi Token Prediction" note, K=3 flow step 2 (stacked queries against the
// reused cache, causal within the verify chain) in the absorbed MLA form: one
// latent vector of 576 per token is the key, its first 512 entries the value;
// every query head attends it. Row of verify token j (request context ctx)
// attends slots 0..ctx+j.
//
// Transposed formulation so that every operand fits the tensor memory:
//   S^T [128 keys x 64 rows]  = K_tile [128 x 576] . Q^T        (M = keys)
//   O^T [512 dv   x 64 rows] += V^T [dv x 128 keys] . P^T         (M = 128 dv, 4 chunks)
// TMEM: O^T in columns 0..255 (4 chunks x 64), two S^T buffers in 256..383.
// Shared memory holds the Q tile (64 rows x 576, 72 KB) and the whole key
// tile: nine 16 KB slots, slot c = [128 keys x 64 dims] for dims 64c..64c+63.
// QK reads them K-major; PV reads V^T MN-major straight from slots 2dc and
// 2dc+1 (the value is the first 512 latent dims), so the cache is read once.
// P^T (bf16) is written into the rope slot (dims 512..575) once QK is done.
// Slots are released as PV stops needing them and refilled with the next
// tile (prefetched into L2 one tile ahead), so loads overlap PV.
//
// This single-CTA form serves requests whose 64-row blocks do not pair up
// (an odd count); each CTA fetches its own copy of every key tile.
//
// Warps (5 warpgroups): 0 MMA issuer, 1-3 TMA producers (lanes 0 and 1 of
// each issue one 8 KB box at a time, so six copies stay in flight), 4..19
// softmax / epilogue (warp w owns TMEM lanes 32*(w%4)..+31 = keys of S^T, dv
// of O^T, and one quarter of the 64 row columns). setmaxnreg moves registers
// from warpgroup 0 to the softmax warpgroups.
//
// Online softmax with a lazy rescale: the reference row max only moves when
// a score exceeds it by more than 8 (log2 units); one barrier reduction tells
// all softmax warps whether any did, and only then are the tile's row maxima
// taken (butterfly transpose-reduce over the warp plus a 4-way merge in shared
// memory) and the O^T columns rescaled. Results are exact either way since P
// and l use the same reference. Each thread keeps partial row sums over its
// keys; they are reduced once, after the last tile.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mtp {

bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box);

namespace {

constexpr int kRows = 64;             // query rows per CTA (MMA N)
constexpr int kKeys = 128;            // keys per tile (MMA M of S^T)
constexpr int kDQ = 576, kDV = 512;
constexpr int kQChunks = kDQ / 64;    // 9
constexpr int kSlotBytes = 16384;     // one [128 keys x 64 dims] chunk of the tile
constexpr int kSlots = kQChunks;      // the whole tile is resident: slot c = dims 64c .. 64c+63
constexpr int kPSlot = 8;             // the rope chunk's slot receives P^T once QK is done
constexpr int kSBufs = 2;
constexpr int kSoftWarps = 16;        // 4 per TMEM lane quarter, 16 row columns each
constexpr int kProducers = 6;         // TMA issuing warps (warps 1-3 and 13-15)         // 2 per TMEM lane quarter (row halves)
constexpr int kThreads = 640;         // 5 warpgroups: [MMA, producer x 3], softmax x 4
constexpr int kLaunchRegs = 96;       // registers per thread at launch (65536 / 640, rounded down to 8)
constexpr int kRegsLight = 56;        // MMA / producer warpgroup after setmaxnreg
constexpr int kRegsSoftmax = 104;     // softmax warpgroups
static_assert(128 * kRegsLight + 4 * 128 * kRegsSoftmax <= kThreads * kLaunchRegs,
              "register split exceeds the registers the block is launched with");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyRescale = 8.0f;  // log2 units

constexpr int kQOff = 0;                                    // 9 x 8 KB
constexpr int kSlotOff = kQOff + kQChunks * 8192;           // 73728
constexpr int kRedOff = kSlotOff + kSlots * kSlotBytes;     // red_max[4][64], red_sum[4][64]
constexpr int kRowOff = kRedOff + 2 * 4 * 64 * 4;           // m_run, l_run, m_ref, scale [64] floats, path [64] u32, shift [64]
constexpr int kBarOff = kRowOff + 6 * 64 * 4;
constexpr int kNumBars = 2 * kSlots + 1 + 2 * kSBufs + 1 + 1 + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;            // tmem base, abort, rescale flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;       // O^T chunk c at c * 64
constexpr uint32_t kColS = 256;     // S^T buffer b at 256 + b * 64

struct Params {
  __nv_bfloat16* out;
  float* part_o;
  float* part_lse;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* order;   // work items, longest first (mla_schedule_kernel)
  const int32_t* parents; // [B, R] tree drafts, nullptr: chains
  unsigned* err;
  int B, R, Hq, max_blocks, num_blocks, split_len, n_splits;
  int groups;           // work groups per request: row blocks (single CTA) or row-block pairs (CTA pairs)
  int cluster;          // CTAs per work group: 1, or 2 for the CTA-pair kernel
  int n_items;          // work items in the order (the persistent CTA-pair kernel walks them)
  float scale_log2;
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return sm100::smem_desc_sw128_kmajor(saddr); }

// MN-major operand with 128-B swizzling: 64-element MN blocks `lbo` bytes
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

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void softmax_barrier() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Named barrier 1 over the 512 softmax threads that also returns whether any
// of them passed true.
__device__ __forceinline__ bool softmax_barrier_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, 1, 512, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
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

// Two floats to bf16 (round to nearest even) in one instruction: lo in bits
// 0..15, hi in bits 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void store_b16(uint8_t* p, uint32_t v) {
  *reinterpret_cast<uint16_t*>(p) = (uint16_t)v;
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Lane l ends up with op-reduction over the 32 lanes of element l of v[]
// (a butterfly transpose-reduce: 31 shuffles for 32 values).
template <bool kMax>
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = upper ? v[k] : v[k + w];
      const float keep = upper ? v[k + w] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// A work item is (split, request, group g of C row blocks): item index
// i = (split * B + b) * groups + g. Every CTA of the group walks the keys
// [t0, t_end) visible to the group's last row.
struct Item {
  int split, b, g;
};

__device__ __forceinline__ Item decode_item(int i, int B, int groups) {
  Item it;
  it.g = i % groups;
  it.b = (i / groups) % B;
  it.split = i / (groups * B);
  return it;
}

__device__ __forceinline__ int item_key_end(const Item& it, int ctx, int R, int Hq, int rows, int C, int split_len) {
  const int cluster_rows_end = min((it.g + 1) * C * kRows, rows);
  const int j_max = min(R - 1, (cluster_rows_end - 1) / Hq);
  return min(it.split * split_len + split_len, ctx + j_max + 1);
}

constexpr int kMaxItemTiles = 64;   // split_len <= 8192 keys = 64 tiles

// Orders the work items by tile count, longest first (counting sort, one
// CTA). Clusters are dispatched in index order, so long items start first
// and short ones fill the tail.
__global__ void __launch_bounds__(1024) mla_schedule_kernel(const int32_t* __restrict__ ctx_lens, int B, int R, int Hq,
                                                           int C, int groups, int split_len, int n_splits,
                                                           int max_len, int32_t* __restrict__ order) {
  __shared__ int hist[kMaxItemTiles + 1];
  const int rows = R * Hq, n = n_splits * B * groups;
  auto tiles_of = [&](int i) -> int {
    const Item it = decode_item(i, B, groups);
    const int ctx = ctx_lens[it.b];
    if (ctx < 0 || ctx + R > max_len) return 0;   // rejected by the attention kernel itself
    const int t0 = it.split * split_len;
    const int t_end = item_key_end(it, ctx, R, Hq, rows, C, split_len);
    return t0 < t_end ? min((t_end - t0 + kKeys - 1) / kKeys, kMaxItemTiles) : 0;
  };
  for (int k = threadIdx.x; k <= kMaxItemTiles; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&hist[tiles_of(i)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {   // hist[k] becomes the first position of tile count k
    int acc = 0;
    for (int k = kMaxItemTiles; k >= 0; --k) {
      const int h = hist[k];
      hist[k] = acc;
      acc += h;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) order[atomicAdd(&hist[tiles_of(i)], 1)] = i;
}

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

// kTree: rows see the verify keys of their root path (tree drafts); the chain
// instantiation keeps each row's plain key limit ctx + j in the same array.
template <bool kTree>
__global__ void __launch_bounds__(kThreads, 1) attn_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                  const __grid_constant__ CUtensorMap tm_kv,
                                                                  const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red_max = reinterpret_cast<float*>(smem + kRedOff);
  float* red_sum = red_max + 4 * 64;
  float* m_run = reinterpret_cast<float*>(smem + kRowOff);
  float* l_run = m_run + 64;
  float* m_ref = m_run + 128;
  float* rscale = m_run + 192;
  uint32_t* path = reinterpret_cast<uint32_t*>(m_run + 256);   // per row: path mask (tree) or key limit (chain)
  float* m_shift = m_run + 320;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);   // [kSlots]: slot c holds this tile's chunk c
  uint64_t* empty = full + kSlots;                                  // [kSlots]: the MMAs are done with it
  uint64_t* qbar = empty + kSlots;
  uint64_t* s_full = qbar + 1;
  uint64_t* s_empty = s_full + kSBufs;
  uint64_t* p_full = s_empty + kSBufs;
  uint64_t* o_done = p_full + 1;
  uint64_t* final_bar = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int C = 1;   // one row block per work item
  const Item item = decode_item(p.order[blockIdx.x], p.B, p.groups);
  const int split = item.split, b = item.b;
  const int rows = p.R * p.Hq;
  const int row_base = item.g * kRows;
  const int ctx = p.ctx_lens[b];
  if (ctx < 0 || ctx + p.R > p.max_blocks * kBlock) {
    if (threadIdx.x == 0 && split == 0 && row_base == 0) raise_error(p.err, MTP_ERR_LENGTH);
    return;
  }
  // The CTA walks the keys visible to its last row; rows that see fewer keys
  // mask the rest.
  const int t0 = split * p.split_len;
  const int t_end = item_key_end(item, ctx, p.R, p.Hq, rows, C, p.split_len);
  if (t0 >= t_end) return;  // no key of this split is visible to these rows: the combine skips it
  const int n_tiles = (t_end - t0 + kKeys - 1) / kKeys;

  if (threadIdx.x == 0) {
    for (int c = 0; c < kSlots; ++c) {
      sm100::mbar_init(&full[c], 2);   // one arrival per box
      sm100::mbar_init(&empty[c], 1);
    }
    sm100::mbar_init(qbar, 1);
    for (int i = 0; i < kSBufs; ++i) {
      sm100::mbar_init(&s_full[i], 1);
      sm100::mbar_init(&s_empty[i], kSoftWarps);
    }
    sm100::mbar_init(p_full, kSoftWarps);
    sm100::mbar_init(o_done, 1);
    sm100::mbar_init(final_bar, 1);
    *abort = 0;
    sm100::fence_barrier_init();
  }
  if (warp == 0) {
    sm100::tmem_alloc(tmem_slot, kTmemCols);
    sm100::tmem_relinquish();
  }
  if (threadIdx.x < kRows) {
    const int rr = min(row_base + (int)threadIdx.x, rows - 1);
    path[threadIdx.x] = kTree ? tree_path_mask(p.parents, b, p.R, rr / p.Hq, p.err) : (uint32_t)(ctx + rr / p.Hq);
    m_run[threadIdx.x] = -INFINITY;
    m_ref[threadIdx.x] = 0.0f;   // reference max the softmax warps start from
    l_run[threadIdx.x] = 0.0f;
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = sm100::smem_u32(smem);
  const uint32_t p_base = smem_base + kSlotOff + kPSlot * kSlotBytes;

  auto softmax_role = [&]() {
    // ------------------------------------------------------- softmax warps
    const int sw = warp - 4;                 // 0..15
    const int qq = warp % 4;                 // TMEM lane quarter: keys / dv 32*qq + lane
    const int cq = sw >> 2;                  // row quarter: rows 16*cq .. 16*cq+15
    const int st = sw * 32 + lane;           // 0..511
    const uint32_t lane_addr = (uint32_t)(32 * qq) << 16;
    // Thread (qq, lane) sees key 32*qq + lane of every tile for the 16 rows of
    // its quarter and keeps its own partial row sums; the sums are reduced
    // over the keys once, after the last tile.
    float acc[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) acc[x] = 0.0f;
    // first key some row of the block may not see: after the first row's own key for a chain, the
    // first verify key for a tree
    const int mask_from = kTree ? ctx : ctx + row_base / p.Hq + 1;
    // Every softmax warp runs the same sequence of named barriers for every
    // tile; after an abort the tensor-memory work is skipped but the barrier
    // sequence is kept, so no warp is left waiting on the others.
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % kSBufs;
      // S^T(i) is complete; so is every earlier MMA, PV(i-1) included (the
      // tile's rope chunk was refilled only after PV(i-1) released its slot).
      ok = ok && __all_sync(0xffffffffu, sm100::mbar_wait(&s_full[buf], (i / kSBufs) & 1, abort) ? 1 : 0);
      // d = score (log2 units) - reference max of the row.
      float d[16];
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
      // The reference only moves when a score exceeds it by more than
      // kLazyRescale: then (and on the first tile) the tile's row maxima are
      // taken and the references updated.
      bool exceed = (i == 0);
#pragma unroll
      for (int x = 0; x < 16; ++x) exceed |= d[x] > kLazyRescale;
      if (softmax_barrier_any(exceed)) {
        {
          float t[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) t[x] = d[x];
          // max of d over the warp's keys; the reference is the same for all of them
          const float mx = transpose_reduce16<true>(t, lane);
          if (lane < 16) red_max[qq * 64 + cq * 16 + lane] = mx + m_ref[cq * 16 + lane];
        }
        softmax_barrier();
        if (st < kRows) {
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
        softmax_barrier();
        bool rescale = false;
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float sc = rscale[cq * 16 + x];
          rescale |= sc != 1.0f;
          acc[x] *= sc;
          d[x] += m_shift[cq * 16 + x];
        }
        // O^T columns of these rows hold PV up to tile i-1 (complete): rescale them.
        if (ok && i > 0 && rescale) {
#pragma unroll 1
          for (int dc = 0; dc < 4; ++dc) {
            uint32_t r[16];
            const uint32_t ta = tmem + lane_addr + kColO + dc * 64 + cq * 16;
            tmem_ld_32x32b_x16(ta, r);
            sm100::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * rscale[cq * 16 + x]);
            tmem_st_32x32b_x16(ta, r);
          }
          tmem_st_wait();
        }
      }
      // p = 2^d: P^T (bf16) into the rope slot as a K-major B tile (block of
      // 64 keys, row, key), and into this thread's partial row sums.
      {
        const int k = 32 * qq + lane;
        uint8_t* pb = smem + kSlotOff + kPSlot * kSlotBytes + (k >> 6) * 8192;
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
      if (lane == 0 && ok) sm100::mbar_arrive(p_full);
    }
    if (!ok && lane == 0) {
      *abort = 1;
      raise_error(p.err, MTP_ERR_TIMEOUT);
    }
    // Row sums: over the warp's 32 keys, then over the 4 lane quarters.
    {
      const float sm = transpose_reduce16<false>(acc, lane);
      if (lane < 16) red_sum[qq * 64 + cq * 16 + lane] = sm;
    }
    softmax_barrier();
    if (st < kRows) l_run[st] = red_sum[st] + red_sum[64 + st] + red_sum[128 + st] + red_sum[192 + st];
    // -------------------------------------------------------- epilogue
    const bool done = ok && __all_sync(0xffffffffu, sm100::mbar_wait(o_done, (n_tiles - 1) & 1, abort) ? 1 : 0);
    softmax_barrier();
    if (done) {
      sm100::tc_fence_after();
      const int dvl = 32 * qq + lane;
#pragma unroll 1
      for (int dc = 0; dc < 4; ++dc) {
        const int dv = dc * 128 + dvl;
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem + lane_addr + kColO + dc * 64 + cq * 16, r);
        sm100::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int rloc = cq * 16 + x;
          const int rr = row_base + rloc;
          if (rr >= rows) continue;
          const float l = l_run[rloc];
          const float o = l > 0.0f ? __uint_as_float(r[x]) / l : 0.0f;
          const int64_t orow = (int64_t)b * rows + rr;
          if (p.n_splits == 1) p.out[orow * kDV + dv] = __float2bfloat16_rn(o);
          else p.part_o[(orow * p.n_splits + split) * kDV + dv] = o;
        }
      }
      if (p.n_splits > 1 && st < kRows && row_base + st < rows) {
        const float l = l_run[st];
        const int64_t orow = (int64_t)b * rows + row_base + st;
        p.part_lse[orow * p.n_splits + split] = l > 0.0f ? (m_run[st] + log2f(l)) * kLn2 : -INFINITY;
      }
    }
  };

  // Warp roles. Warpgroups 0 and 3 hand registers to the softmax warpgroups
  // (every warp of a warpgroup runs the same setmaxnreg).
  const int wg = warp / 4;
  if (wg >= 1) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    softmax_role();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLight));
    const int pw = (warp >= 1 && lane < 2) ? 2 * (warp - 1) + lane : -1;   // producer 0..5 (warps 1-3, lanes 0-1)
    if (pw >= 0) {
      // ------------------------------------------------------ TMA producers
      // A tile is 18 boxes of [64 keys x 64 dims] (8 KB): box x = slot x/2,
      // keys 64*(x%2).. of the tile. Producer pw owns boxes pw, pw+6, pw+12
      // (slots in the order the MMA consumes them) and refills a box as soon
      // as the MMAs released its slot from the previous tile. Each
      // box issue is followed by an L2 prefetch of the same box of the next
      // tile, so that the refill after the release hits L2.
      const uint64_t pol_kv = sm100::l2_policy_evict_last();   // the request's other row blocks re-read it
      if (pw == 0) {
        sm100::tma_prefetch_desc(&tm_q);
        sm100::tma_prefetch_desc(&tm_kv);
        sm100::mbar_arrive_expect_tx(qbar, kQChunks * 8192);
        const uint64_t pol_q = sm100::l2_policy_evict_first();
        for (int c = 0; c < kQChunks; ++c)
          sm100::tma_load_2d(smem + kQOff + c * 8192, &tm_q, qbar, c * 64, b * rows + row_base, pol_q);
      }
      const int32_t* tbl = p.block_table + (int64_t)b * p.max_blocks;
      auto block_of = [&](int key0) -> int {   // cache block holding keys key0..key0+63, or -1 (zero fill)
        if (key0 >= t_end) return -1;
        const int blk = tbl[key0 / kBlock];
        if (blk < 0 || blk >= p.num_blocks) {
          raise_error(p.err, MTP_ERR_BLOCK_ID);
          return -1;
        }
        return blk;
      };
      bool ok = true;
      for (int i = 0; i < n_tiles && ok; ++i) {
#pragma unroll 1
        for (int x = pw; x < 2 * kSlots; x += kProducers) {
          const int c = x >> 1, half = x & 1;
          ok = sm100::mbar_wait(&empty[c], (uint32_t)((i & 1) ^ 1), abort);
          if (!ok) break;
          sm100::mbar_arrive_expect_tx(&full[c], kSlotBytes / 2);
          const int blk = block_of(t0 + i * kKeys + half * 64);
          uint8_t* dst = smem + kSlotOff + c * kSlotBytes + half * (kSlotBytes / 2);
          sm100::tma_load_3d(dst, &tm_kv, &full[c], c * 64, 0, blk, pol_kv);
          if (i + 1 < n_tiles) {
            const int nblk = block_of(t0 + (i + 1) * kKeys + half * 64);
            if (nblk >= 0) sm100::tma_prefetch_3d(&tm_kv, c * 64, 0, nblk);
          }
        }
      }
      if (!ok) {
        *abort = 1;
        raise_error(p.err, MTP_ERR_TIMEOUT);
      }
      // Every copy must land before the CTA may exit: wait (time-limited)
      // for the last fill of each slot this producer fed.
      if (pw == 0) sm100::mbar_wait_timeout(qbar, 0, sm100::kWaitTimeoutNs);
      for (int x = pw; x < 2 * kSlots; x += kProducers)
        sm100::mbar_wait_timeout(&full[x >> 1], (uint32_t)((n_tiles - 1) & 1), sm100::kWaitTimeoutNs);
    } else if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- MMA
      // QK(i) over the 9 resident chunks, then (once P(i) is published) PV(i)
      // reading V^T MN-major from chunk slots 2dc, 2dc+1 and P^T from the rope
      // slot; each slot is released to the producers as soon as PV(i) no
      // longer needs it, so tile i+1 loads overlap PV(i). Descriptors are
      // formed once and advanced by constants (16-byte units in the start
      // address field): the issue loop must stay far below one MMA's time.
      constexpr uint32_t idesc_qk = sm100::idesc_bf16_f32(128, kRows);
      constexpr uint32_t idesc_pv = sm100::idesc_bf16_f32(128, kRows) | (1u << 15);   // A (V^T) MN-major
      const uint64_t d_slot = desc_kmajor(smem_base + kSlotOff);
      const uint64_t d_q = desc_kmajor(smem_base + kQOff);
      const uint64_t d_vt = desc_mnmajor(smem_base + kSlotOff, kSlotBytes);
      const uint64_t d_p = desc_kmajor(p_base);
      auto release = [&](int c) { sm100::tc_commit(&empty[c]); };
      bool ok = sm100::mbar_wait(qbar, 0, abort);
      auto issue_qk = [&](int i) -> bool {
        const int buf = i % kSBufs;
        if (!sm100::mbar_wait(&s_empty[buf], ((i / kSBufs) & 1) ^ 1u, abort)) return false;
        sm100::tc_fence_after();
        const uint32_t d = tmem + kColS + buf * 64;
#pragma unroll 1
        for (int c = 0; c < kSlots; ++c) {
          if (!sm100::mbar_wait(&full[c], (uint32_t)(i & 1), abort)) return false;
          sm100::tc_fence_after();
          const uint64_t a = d_slot + (uint64_t)(c * (kSlotBytes >> 4));
          const uint64_t q = d_q + (uint64_t)(c * (8192 >> 4));
          sm100::tc_mma_bf16(d, a, q, idesc_qk, c > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) sm100::tc_mma_bf16(d, a + 2 * kk, q + 2 * kk, idesc_qk, 1u);
        }
        sm100::tc_commit(&s_full[buf]);
        return true;
      };
      auto issue_pv = [&](int i) -> bool {
        if (!sm100::mbar_wait(p_full, (uint32_t)(i & 1), abort)) return false;
        sm100::tc_fence_after();
        const uint32_t first = i > 0 ? 1u : 0u;
#pragma unroll 1
        for (int dc = 0; dc < 4; ++dc) {
          const uint64_t a = d_vt + (uint64_t)(2 * dc * (kSlotBytes >> 4));
          const uint32_t d = tmem + kColO + dc * 64;
          sm100::tc_mma_bf16(d, a, d_p, idesc_pv, first);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            sm100::tc_mma_bf16(d, a + (uint64_t)(kk * (2048 >> 4)),
                               d_p + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_pv, 1u);
          release(2 * dc);
          release(2 * dc + 1);
        }
        release(kPSlot);
        sm100::tc_commit(o_done);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int i = 0; i < n_tiles && ok; ++i) {
        ok = issue_pv(i);
        if (ok && i + 1 < n_tiles) ok = issue_qk(i + 1);
      }
      if (!ok) {
        *abort = 1;
        raise_error(p.err, MTP_ERR_TIMEOUT);
      }
      sm100::tc_commit(final_bar);
      sm100::mbar_wait_timeout(final_bar, 0, sm100::kWaitTimeoutNs);
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// CTA-pair variant (tcgen05 cta_group::2): the two CTAs of a cluster hold 64
// query rows each (two row blocks of one request) and share every MMA:
//   S [128 rows x 128 keys]   = Q . K^T   pair M = 128 (64 rows per CTA), N = 128 keys;
//                                           each CTA stages 64 of the tile's keys, all 576 dims
//   O [128 rows x 512 dv]    += P . V     pair M = 128, N = 256 dv, twice (dv 0..255, 256..511);
//                                           each CTA stages V of all 128 keys for its 128-dv
//                                           half of each product (B operand, MN-major)
// Each CTA's TMEM then holds S and O of its own 64 rows only (TMEM lane l: row
// l % 64; lanes 64..127 carry the second half of the columns), so the softmax,
// its lazy rescale, the row sums and the normalisation stay local to the CTA.
// Per 128-key tile a CTA stages 136 KB and reads ~250 KB of operands, against
// 147 KB and ~410 KB for one 64-row CTA on its own; the MMAs have N = 128/256.
// The key tile is single-buffered, so the next tile's keys can only load into
// chunks that QK has finished with: the nine K chunks land and are released
// in three groups of three, and the eight V boxes in four quarters (key half
// x dv half, PV's four quarters in turn), so the loads of tile i+1 start
// while QK(i) and PV(i) still run. Two warps issue the MMAs: one QK(i) as
// soon as its key groups land, the other PV(i) as soon as P(i) is written, so
// QK(i+1) runs during the softmax of tile i instead of waiting behind PV(i)
// (S is double-buffered; each issuing warp waits only for its own inputs: a
// wait costs the issuing warp a few hundred clocks even when the phase is
// already complete). P is single-buffered: the softmax of tile i computes its
// probabilities in registers, then waits for PV(i-1) before writing them (and
// before using the reduction scratch, which shares the P buffer).
// The pairs are persistent (one per resident cluster slot) and walk several
// work items each; the barrier phases run on across items, the next item's Q
// and first tiles load while the current one ends, and its first PV waits
// only for the epilogue to have read O out. The epilogue stages the output
// through the P buffer so that it leaves as whole 128-byte lines.
namespace pr {
constexpr int kQOff = 0;                          // 9 x [64 rows x 64 dims]
constexpr int kKOff = kQOff + 9 * 8192;           // 9 x [64 own keys x 64 dims]
constexpr int kVOff = kKOff + 9 * 8192;           // 8 x [64 keys x 64 dv]: slot (h * 2 + kb) * 2 + j
constexpr int kPOff = kVOff + 8 * 8192;           // P [64 rows x 128 keys]: keys 0..63, then 64..127
constexpr int kRedOff = kPOff + 8192;             // red_max[8][64], red_sum[8][64] alias P keys 64..127
constexpr int kRowOff = kPOff + 2 * 8192;         // m_run, m_ref, rscale, m_shift, l_run [64] f32 (+ 64 spare)
constexpr int kBarOff = kRowOff + 6 * 64 * 4;
constexpr int kKGroups = 3;                       // the nine K chunks land and are released in this many groups
constexpr int kKPerGroup = 9 / kKGroups;
static_assert(kKGroups * kKPerGroup == 9, "K groups must split the nine chunks evenly");
constexpr int kNumBars = 2 * kKGroups + 4 + 4 + 2 + 2 + 2 + 1 + 1 + 1 + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM base, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
constexpr uint32_t kColO = 0;                     // O of product h at columns 128 h .. +127
constexpr uint32_t kColS = 256;                   // S buffer b at 256 + 64 b
}  // namespace pr

template <bool kTree>
__global__ void __launch_bounds__(kThreads, 1) attn_mla_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                    const __grid_constant__ CUtensorMap tm_kv,
                                                                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red_max = reinterpret_cast<float*>(smem + pr::kRedOff);   // [8][64]
  float* red_sum = red_max + 8 * 64;
  float* m_run = reinterpret_cast<float*>(smem + pr::kRowOff);
  float* m_ref = m_run + 64;
  float* rscale = m_run + 128;
  float* m_shift = m_run + 192;
  float* l_run = m_run + 256;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + pr::kBarOff);   // [3] leader: both CTAs' K chunk group landed
  uint64_t* kempty = kfull + pr::kKGroups;                              // [3] both: the group's K slots are free
  uint64_t* vfull = kempty + pr::kKGroups;                              // [4] leader: both CTAs' V boxes of a quarter
  uint64_t* vempty = vfull + 4;                                         // [4] both: the quarter's V slots are free
  uint64_t* qbar = vempty + 4;                                          // leader: both CTAs' Q of an item landed
  uint64_t* qempty = qbar + 1;                                          // both: an item's last QK read Q
  uint64_t* s_full = qempty + 1;                                        // [2] both
  uint64_t* s_empty = s_full + 2;                                       // [2] leader, one arrive per CTA
  uint64_t* p_full = s_empty + 2;                                       // leader, one arrive per CTA
  uint64_t* o_done = p_full + 1;                                        // both
  uint64_t* o_free = o_done + 1;                                        // leader, one arrive per CTA: O read out
  uint64_t* final_bar = o_free + 1;                                     // both
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + pr::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + pr::kMiscOff + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = sm100::cluster_ctarank();
  const bool leader = rank == 0;
  const int rows = p.R * p.Hq;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  // The pair's work items: round k takes order slot k * n_pairs + pair, or
  // its mirror image for odd k, so the longest items (first in the order)
  // share a pair with the shortest ones. Every role walks the same list.
  struct Work {
    int split, b, row_base, ctx, t0, t_end, n_tiles;
    bool bad_len;
  };
  auto work = [&](int k, Work& w) -> bool {
    const int slot = k * n_pairs + ((k & 1) ? n_pairs - 1 - pair : pair);
    if (slot >= p.n_items) return false;
    const Item it = decode_item(p.order[slot], p.B, p.groups);
    w.split = it.split;
    w.b = it.b;
    w.row_base = (it.g * 2 + (int)rank) * kRows;
    w.ctx = p.ctx_lens[it.b];
    w.t0 = it.split * p.split_len;
    w.t_end = w.t0;
    w.n_tiles = 0;
    w.bad_len = w.ctx < 0 || w.ctx + p.R > p.max_blocks * kBlock;   // uniform over the pair (same request)
    if (!w.bad_len) {
      w.t_end = item_key_end(it, w.ctx, p.R, p.Hq, rows, 2, p.split_len);
      if (w.t0 < w.t_end) w.n_tiles = (w.t_end - w.t0 + kKeys - 1) / kKeys;
    }
    return true;
  };

  if (threadIdx.x == 0) {
    for (int g = 0; g < pr::kKGroups; ++g) {
      sm100::mbar_init(&kfull[g], 1);
      sm100::mbar_init(&kempty[g], 1);
    }
    for (int k = 0; k < 4; ++k) {
      sm100::mbar_init(&vfull[k], 1);
      sm100::mbar_init(&vempty[k], 1);
    }
    for (int k = 0; k < 2; ++k) {
      sm100::mbar_init(&s_full[k], 1);
      sm100::mbar_init(&s_empty[k], 2);   // one arrive per CTA
    }
    sm100::mbar_init(qbar, 1);
    sm100::mbar_init(qempty, 1);
    sm100::mbar_init(p_full, 2);
    sm100::mbar_init(o_done, 1);
    sm100::mbar_init(o_free, 2);
    sm100::mbar_init(final_bar, 2);   // the QK and the PV issuer each commit once at the end
    *abort = 0;
    sm100::fence_barrier_init();
  }
  if (warp == 0) {
    sm100::tmem_alloc_pair(tmem_slot, kTmemCols);
    sm100::tmem_relinquish_pair();
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::cluster_sync();   // both CTAs' barriers and TMEM exist before any remote arrive, load or MMA
  sm100::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = sm100::smem_u32(smem);

  auto softmax_role = [&]() {
    // ------------------------------------------------------- softmax warps
    // Warp (q = warp % 4, sub = (warp - 4) / 4): TMEM lanes 32 q .. 32 q + 31,
    // i.e. rows r = 32 (q % 2) + lane, keys 64 (q / 2) + 16 sub .. + 15 of S.
    const int sw = warp - 4;
    const int q = warp % 4, sub = sw >> 2;
    const int r = 32 * (q & 1) + lane;
    const int khalf = q >> 1;
    const int part = khalf * 4 + sub;                 // which of the row's 8 partials this thread holds
    const int st = sw * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    bool ok = true;
    int T = 0;                                        // tiles of this pair before the current item
    Work w, wn;
    bool has = work(0, w);
    for (int k = 0; has; ++k, w = wn) {
      has = work(k + 1, wn);   // the next item's record loads while this one runs
      if (w.n_tiles == 0) {
        if (w.bad_len && st == 0 && w.split == 0 && w.row_base == 0) raise_error(p.err, MTP_ERR_LENGTH);
        continue;
      }
      const int rr0 = min(w.row_base + r, rows - 1);
      const uint32_t path_r = kTree ? tree_path_mask(p.parents, w.b, p.R, rr0 / p.Hq, p.err)
                                    : (uint32_t)(w.ctx + rr0 / p.Hq);   // root-path mask, or the key limit
      const int mask_from = kTree ? w.ctx : w.ctx + w.row_base / p.Hq + 1;   // first key some row may not see
      if (st < kRows) {
        m_run[st] = -INFINITY;
        m_ref[st] = 0.0f;
      }
      softmax_barrier();
      float acc = 0.0f;                               // partial row sum over this thread's keys
      for (int i = 0; i < w.n_tiles; ++i) {
        const int ti = T + i;                         // the pair's tile counter sets the barrier phases
        const int buf = ti & 1;
        ok = ok && __all_sync(0xffffffffu, sm100::mbar_wait_cluster(&s_full[buf], (ti >> 1) & 1, abort) ? 1 : 0);
        float d[16];
        const float mr = m_ref[r];
        if (ok) {
          sm100::tc_fence_after();
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_addr + pr::kColS + buf * 64 + sub * 16, v);
          sm100::tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x) d[x] = fmaf(__uint_as_float(v[x]), p.scale_log2, -mr);
          sm100::tc_fence_before();
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) d[x] = -INFINITY;
        }
        const int tile0 = w.t0 + i * kKeys;
        if (tile0 + kKeys - 1 >= mask_from || tile0 + kKeys > w.t_end) {   // causal / split edge inside the tile
          const int key0 = tile0 + 64 * khalf + 16 * sub;
#pragma unroll
          for (int x = 0; x < 16; ++x)
            d[x] = (key0 + x >= w.t_end || (kTree ? tree_hidden(key0 + x, w.ctx, path_r) : key0 + x > (int)path_r))
                       ? -INFINITY
                       : d[x];
        }
        bool exceed = (i == 0);
#pragma unroll
        for (int x = 0; x < 16; ++x) exceed |= d[x] > kLazyRescale;
        const bool any_exceed = softmax_barrier_any(exceed);
        // every softmax warp of this CTA has read S from TMEM: one arrive
        if (st == 0) sm100::mbar_arrive_remote_relaxed(&s_empty[buf], 0);
        // The previous PV reads P (which the reduction scratch shares) and
        // accumulates into O, and may still run (QK does not wait for it): the
        // O rescale and the P stores wait for its completion. (The softmax of
        // the previous tile waited for the PV before it, so the parity cannot
        // alias an older phase; before an item's first tile the previous
        // item's epilogue has already waited for its last PV.)
        bool pv_done = i == 0;
        auto wait_pv = [&]() {
          if (!pv_done) {
            ok = ok && __all_sync(0xffffffffu, sm100::mbar_wait_cluster(o_done, (ti - 1) & 1, abort) ? 1 : 0);
            sm100::tc_fence_after();
            pv_done = true;
          }
        };
        if (any_exceed) {
          wait_pv();
          float mx = d[0];
#pragma unroll
          for (int x = 1; x < 16; ++x) mx = fmaxf(mx, d[x]);
          red_max[part * 64 + r] = mx + mr;
          softmax_barrier();
          if (st < kRows) {
            float mt = red_max[st];
#pragma unroll
            for (int j = 1; j < 8; ++j) mt = fmaxf(mt, red_max[j * 64 + st]);
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
          softmax_barrier();
          const float sc = rscale[r];
          acc *= sc;
          const float sh = m_shift[r];
#pragma unroll
          for (int x = 0; x < 16; ++x) d[x] += sh;
          // O of these rows holds PV up to the previous tile (complete): rescale
          // it. This warp owns 64 of the 256 O columns of its TMEM lanes.
          if (ok && i > 0 && __any_sync(0xffffffffu, sc != 1.0f)) {
            const int h = sub >> 1, c0 = (sub & 1) * 64;
#pragma unroll 1
            for (int t = 0; t < 4; ++t) {
              uint32_t v[16];
              const uint32_t ta = tmem + lane_addr + pr::kColO + h * 128 + c0 + t * 16;
              tmem_ld_32x32b_x16(ta, v);
              sm100::tmem_ld_wait();
#pragma unroll
              for (int x = 0; x < 16; ++x) v[x] = __float_as_uint(__uint_as_float(v[x]) * sc);
              tmem_st_32x32b_x16(ta, v);
            }
            tmem_st_wait();
          }
        }
        // p = 2^d into P [64 rows x 128 keys] (K-major A operand of PV, two
        // 64-key blocks) and into the partial row sum, once the previous PV is
        // complete (no thread reads red_max any more, which shares the second
        // block).
        {
          uint8_t* pb = smem + pr::kPOff + khalf * 8192 + r * 128;
          uint32_t wv[8];
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const float p0 = fast_exp2(d[x]), p1 = fast_exp2(d[x + 1]);
            acc += p0 + p1;
            wv[x / 2] = pack_bf16x2(p0, p1);
          }
          wait_pv();
          const int ch = 2 * sub;   // 16-byte chunks 2 sub, 2 sub + 1 of the row
          *reinterpret_cast<uint4*>(pb + (((ch) ^ (r & 7)) << 4)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          *reinterpret_cast<uint4*>(pb + (((ch + 1) ^ (r & 7)) << 4)) = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
        // Every writer makes its P stores visible to the async proxy, then the
        // named barrier orders all of them before the one arrive; a release at
        // cluster scope would add about a microsecond here (measured) without
        // ordering anything the fence and the barrier have not.
        fence_async_smem();
        sm100::tc_fence_before();
        softmax_barrier();   // all of this CTA's P is written
        if (st == 0 && ok) sm100::mbar_arrive_remote_relaxed(p_full, 0);
      }
      // ------------------------------------------------------ epilogue
      // The item's last PV is complete (so P, which red_sum shares, is free).
      const bool done_w = ok && __all_sync(0xffffffffu, sm100::mbar_wait_cluster(o_done, (T + w.n_tiles - 1) & 1,
                                                                                  abort) ? 1 : 0);
      const bool done = !softmax_barrier_any(!done_w);   // uniform: the stores below use named barriers
      red_sum[part * 64 + r] = acc;
      softmax_barrier();
      if (st < kRows) {
        float l = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) l += red_sum[j * 64 + st];
        l_run[st] = l;
      }
      softmax_barrier();
      if (done) {
        sm100::tc_fence_after();
        const int h = sub >> 1, c0 = (sub & 1) * 64;
        const int rr = w.row_base + r;
        const float l = l_run[r];
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const int dv0 = 256 * h + 128 * khalf + c0;     // this thread's TMEM lane 32 q + lane: dv half q / 2
        if (p.n_splits == 1) {
          // Each thread holds one 128-byte block of its row (64 dv, block
          // dv0 / 64). A thread writing its own row would touch 32 lines per
          // store instruction; instead two blocks of every row at a time go
          // through the P buffer (free now; 16-byte granule g of row r at
          // g ^ (r & 7), conflict-free both ways) and leave as whole lines.
          uint8_t* stage = smem + pr::kPOff;   // [64 rows][256 B]
          const int blk = dv0 >> 6;
          // The thread's 64 values, normalised and packed to bf16 pairs (two
          // TMEM loads in flight per wait).
          uint32_t pk[32];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v0[16], v1[16];
            tmem_ld_32x32b_x16(tmem + lane_addr + pr::kColO + h * 128 + c0 + hh * 32, v0);
            tmem_ld_32x32b_x16(tmem + lane_addr + pr::kColO + h * 128 + c0 + hh * 32 + 16, v1);
            sm100::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; x += 2) {
              pk[hh * 16 + x / 2] = pack_bf16x2(__uint_as_float(v0[x]) * inv, __uint_as_float(v0[x + 1]) * inv);
              pk[hh * 16 + 8 + x / 2] = pack_bf16x2(__uint_as_float(v1[x]) * inv, __uint_as_float(v1[x + 1]) * inv);
            }
          }
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {   // dv blocks 2j, 2j + 1 of every row
            if ((blk >> 1) == j) {
              uint8_t* row = stage + r * 256;
#pragma unroll
              for (int gg = 0; gg < 8; ++gg) {   // 16-byte granules (blk & 1) * 8 + gg of the row's 256 B
                const int g = (blk & 1) * 8 + gg;
                *reinterpret_cast<uint4*>(row + ((g ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * gg], pk[4 * gg + 1], pk[4 * gg + 2], pk[4 * gg + 3]);
              }
            }
            softmax_barrier();
#pragma unroll
            for (int u = 0; u < 2; ++u) {   // 1024 granules: 16 per row, consecutive threads along a row
              const int G = st + 512 * u;
              const int row = G >> 4, g = G & 15;
              if (w.row_base + row < rows) {
                const uint4 val = *reinterpret_cast<const uint4*>(stage + row * 256 + ((g ^ (row & 7)) << 4));
                const int64_t orow = (int64_t)w.b * rows + w.row_base + row;
                *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.out + orow * kDV + 128 * j) + g * 16) = val;
              }
            }
            softmax_barrier();
          }
        } else {
#pragma unroll 1
          for (int t = 0; t < 4; ++t) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(tmem + lane_addr + pr::kColO + h * 128 + c0 + t * 16, v);
            sm100::tmem_ld_wait();
            if (rr < rows) {
              const int64_t orow = (int64_t)w.b * rows + rr;
              float* dst = p.part_o + (orow * p.n_splits + w.split) * kDV + dv0 + t * 16;
#pragma unroll
              for (int x = 0; x < 16; x += 4)
                *reinterpret_cast<float4*>(dst + x) =
                    make_float4(__uint_as_float(v[x]) * inv, __uint_as_float(v[x + 1]) * inv,
                                __uint_as_float(v[x + 2]) * inv, __uint_as_float(v[x + 3]) * inv);
            }
          }
        }
        if (p.n_splits > 1 && st < kRows && w.row_base + st < rows) {
          const float l2 = l_run[st];
          const int64_t orow = (int64_t)w.b * rows + w.row_base + st;
          p.part_lse[orow * p.n_splits + w.split] = l2 > 0.0f ? (m_run[st] + log2f(l2)) * kLn2 : -INFINITY;
        }
      }
      // O is read out (and the row state is free): the PV warp may start the
      // pair's next item, which overwrites O.
      sm100::tc_fence_before();
      softmax_barrier();
      if (st == 0 && ok) sm100::mbar_arrive_remote_relaxed(o_free, 0);
      T += w.n_tiles;
    }
    if (!ok && lane == 0) {
      *abort = 1;
      raise_error(p.err, MTP_ERR_TIMEOUT);
    }
  };

  const int wg = warp / 4;
  if (wg >= 1) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    softmax_role();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLight));
    const int pw = (warp >= 2 && lane < 4) ? 4 * (warp - 2) + lane : -1;   // producer 0..7 (warps 2-3, lanes 0-3)
    if (pw >= 0) {
      // ------------------------------------------------------ TMA producers
      // Per tile a CTA loads 17 boxes of [64 keys x 64 dims]: K chunk c of its
      // own key half (slot c, group c / 3), and V boxes (h, kb, j) = dims
      // 64 (4 h + 2 rank + j) of key half kb. Both CTAs' boxes complete on the
      // leader's barriers. Producers 0-5 own K chunk pw (and pw + 6 for
      // pw < 3), each waiting for its group's slots to be released by the
      // previous tile's QK; producers 6 and 7 own the V boxes of key half
      // pw - 6, quarter (key half, dv half h) by quarter, each released by
      // the previous tile's PV. Producer 0 also loads each item's Q once the
      // previous item's last QK has read the Q buffer, so the next item's
      // loads overlap the end of the current one.
      const uint64_t pol_kv = sm100::l2_policy_evict_last();
      const uint64_t pol_q = sm100::l2_policy_evict_first();
      if (pw == 0) {
        sm100::tma_prefetch_desc(&tm_q);
        sm100::tma_prefetch_desc(&tm_kv);
      }
      constexpr int kGroupBytes = 2 * pr::kKPerGroup * 8192;   // both CTAs' K chunks of a group
      constexpr int kQuarterBytes = 2 * 2 * 8192;              // both CTAs' two V boxes of a quarter
      bool ok = true;
      int T = 0, kq = 0;   // tiles and items with tiles so far
      Work w;
      for (int k = 0; ok && work(k, w); ++k) {
        if (w.n_tiles == 0) continue;
        const int32_t* tbl = p.block_table + (int64_t)w.b * p.max_blocks;
        auto block_of = [&](int key0) -> int {
          if (key0 >= w.t_end) return -1;
          const int blk = tbl[key0 / kBlock];
          if (blk < 0 || blk >= p.num_blocks) {
            raise_error(p.err, MTP_ERR_BLOCK_ID);
            return -1;
          }
          return blk;
        };
        if (pw == 0) {
          if (kq > 0) ok = sm100::mbar_wait_cluster(qempty, (uint32_t)((kq - 1) & 1), abort);
          if (!ok) break;
          if (leader) sm100::mbar_arrive_expect_tx(qbar, 2 * kQChunks * 8192);
          for (int c = 0; c < kQChunks; ++c)   // both CTAs' Q complete on the leader's barrier
            sm100::tma_load_2d_pair(smem + pr::kQOff + c * 8192, &tm_q, qbar, 0, c * 64, w.b * rows + w.row_base,
                                    pol_q);
        }
        for (int i = 0; i < w.n_tiles && ok; ++i) {
          const int ti = T + i;
          const uint32_t par = (uint32_t)((ti & 1) ^ 1);
          if (pw < 6) {
            const int blk = block_of(w.t0 + i * kKeys + 64 * (int)rank);
            for (int c = pw; c < 9; c += 6) {   // chunk pw, then pw + 6 (group 2) for pw < 3
              const int g = c / pr::kKPerGroup;
              ok = sm100::mbar_wait_cluster(&kempty[g], par, abort);
              if (!ok) break;
              if (leader && c % pr::kKPerGroup == 0) sm100::mbar_arrive_expect_tx(&kfull[g], kGroupBytes);
              sm100::tma_load_3d_pair(smem + pr::kKOff + c * 8192, &tm_kv, &kfull[g], 0, c * 64, 0, blk, pol_kv);
            }
          } else {
            const int kb = pw - 6;
            const int blk = block_of(w.t0 + i * kKeys + 64 * kb);
            for (int h = 0; h < 2; ++h) {
              const int qq = kb * 2 + h;
              ok = sm100::mbar_wait_cluster(&vempty[qq], par, abort);
              if (!ok) break;
              if (leader) sm100::mbar_arrive_expect_tx(&vfull[qq], kQuarterBytes);
              for (int j = 0; j < 2; ++j) {
                const int slot = (h * 2 + kb) * 2 + j;
                const int dchunk = 4 * h + 2 * (int)rank + j;
                sm100::tma_load_3d_pair(smem + pr::kVOff + slot * 8192, &tm_kv, &vfull[qq], 0, dchunk * 64, 0, blk,
                                        pol_kv);
              }
            }
          }
        }
        T += w.n_tiles;
        ++kq;
      }
      if (!ok) {
        *abort = 1;
        raise_error(p.err, MTP_ERR_TIMEOUT);
      }
      // The leader's producers wait (time-limited) for the last fill of each
      // barrier they armed; the odd CTA's copies complete on those barriers.
      if (leader && T > 0) {
        const uint32_t last = (uint32_t)((T - 1) & 1);
        if (pw == 0) sm100::mbar_wait_timeout(qbar, (uint32_t)((kq - 1) & 1), sm100::kWaitTimeoutNs);
        if (pw < 6)
          for (int c = pw; c < 9; c += 6)   // the groups this producer armed
            if (c % pr::kKPerGroup == 0)
              sm100::mbar_wait_timeout(&kfull[c / pr::kKPerGroup], last, sm100::kWaitTimeoutNs);
        if (pw >= 6)
          for (int h = 0; h < 2; ++h) sm100::mbar_wait_timeout(&vfull[(pw - 6) * 2 + h], last, sm100::kWaitTimeoutNs);
      }
    } else if (warp <= 1 && leader) {
      // ---------------------------------------------------------------- MMA
      // Warp 0 issues QK group by group as its keys land (S buffer free),
      // warp 1 issues PV once P is written, quarter by quarter as its values
      // land (and, for an item's first tile, once the previous item's O has
      // been read out); each commits its own MMAs. Each whole warp runs its
      // loop (descriptors stay warp-uniform) and one elected lane issues.
      constexpr uint32_t idesc_qk = sm100::idesc_bf16_f32(128, 128);
      constexpr uint32_t idesc_pv = sm100::idesc_bf16_f32(128, 256) | (1u << 16);   // B (V) MN-major
      auto wait_all = [&](uint64_t* bar, uint32_t par) -> bool {
        return __all_sync(0xffffffffu, sm100::mbar_poll_cluster(bar, par, abort) ? 1 : 0) != 0;
      };
      bool ok = true;
      int T = 0, kq = 0;
      Work w;
      if (warp == 0) {
        const uint64_t d_q = desc_kmajor(smem_base + pr::kQOff);
        const uint64_t d_k = desc_kmajor(smem_base + pr::kKOff);
        for (int k = 0; ok && work(k, w); ++k) {
          if (w.n_tiles == 0) continue;
          ok = wait_all(qbar, (uint32_t)(kq & 1));
          for (int i = 0; i < w.n_tiles && ok; ++i) {
            const int ti = T + i;
            const int buf = ti & 1;
            const uint32_t par = (uint32_t)(ti & 1);
            ok = wait_all(&s_empty[buf], ((ti >> 1) & 1) ^ 1u);
            const uint32_t d = tmem + pr::kColS + buf * 64;
            for (int g = 0; g < pr::kKGroups && ok; ++g) {
              ok = wait_all(&kfull[g], par);
              if (!ok) break;
              sm100::tc_fence_after();
              if (sm100::elect_one()) {
#pragma unroll 1
                for (int c = pr::kKPerGroup * g; c < pr::kKPerGroup * (g + 1); ++c) {
                  const uint64_t a = d_q + (uint64_t)(c * 512), bk = d_k + (uint64_t)(c * 512);
                  sm100::tc_mma_bf16_pair(d, a, bk, idesc_qk, c > 0 ? 1u : 0u);
#pragma unroll
                  for (int kk = 1; kk < 4; ++kk) sm100::tc_mma_bf16_pair(d, a + 2 * kk, bk + 2 * kk, idesc_qk, 1u);
                }
                sm100::tc_commit_pair_mc(&kempty[g], 3);   // this group's K slots free once read
                if (g == pr::kKGroups - 1) {
                  sm100::tc_commit_pair_mc(&s_full[buf], 3);
                  if (i == w.n_tiles - 1) sm100::tc_commit_pair_mc(qempty, 3);   // the item's Q is no longer read
                }
              }
              __syncwarp();
            }
          }
          T += w.n_tiles;
          ++kq;
        }
      } else {
        const uint64_t d_p0 = desc_kmajor(smem_base + pr::kPOff);          // P keys 0..63
        const uint64_t d_p1 = desc_kmajor(smem_base + pr::kPOff + 8192);   // P keys 64..127
        const uint64_t d_v = desc_mnmajor(smem_base + pr::kVOff, 8192);
        for (int k = 0; ok && work(k, w); ++k) {
          if (w.n_tiles == 0) continue;
          if (kq > 0) {   // the previous item's O has been read out
            ok = wait_all(o_free, (uint32_t)((kq - 1) & 1));
            if (!ok) break;
            sm100::tc_fence_after();
          }
          for (int i = 0; i < w.n_tiles && ok; ++i) {
            const uint32_t par = (uint32_t)((T + i) & 1);
            ok = wait_all(p_full, par);
            for (int qq = 0; qq < 4 && ok; ++qq) {   // quarter (key half kb, dv half h) = O columns of h over kb's keys
              const int kb = qq >> 1, h = qq & 1;
              ok = wait_all(&vfull[qq], par);
              if (!ok) break;
              sm100::tc_fence_after();
              if (sm100::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  sm100::tc_mma_bf16_pair(tmem + pr::kColO + h * 128, (kb == 0 ? d_p0 : d_p1) + (uint64_t)(kk * 2),
                                          d_v + (uint64_t)(((h * 2 + kb) * 2) * 512 + kk * 128), idesc_pv,
                                          (i > 0 || kb > 0 || kk > 0) ? 1u : 0u);
                sm100::tc_commit_pair_mc(&vempty[qq], 3);   // this quarter's V slots free once read
                if (qq == 3) sm100::tc_commit_pair_mc(o_done, 3);
              }
              __syncwarp();
            }
          }
          T += w.n_tiles;
          ++kq;
        }
      }
      if (!ok && lane == 0) {
        *abort = 1;
        raise_error(p.err, MTP_ERR_TIMEOUT);
      }
      // Every MMA this warp issued has completed before TMEM is released:
      // both issuers commit to the final barrier, warp 0 waits for both.
      if (sm100::elect_one()) sm100::tc_commit_pair_mc(final_bar, 3);
      __syncwarp();
      if (warp == 0) sm100::mbar_wait_timeout(final_bar, 0, sm100::kWaitTimeoutNs);
    } else if (warp == 0 && lane == 0) {
      // odd CTA: the leader's MMAs write this CTA's TMEM; wait for the last one
      sm100::mbar_wait_timeout(final_bar, 0, sm100::kWaitTimeoutNs);
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::cluster_sync();   // neither CTA leaves while the pair's MMAs, copies or arrives may touch it
  if (warp == 0) {
    sm100::tc_fence_after();
    sm100::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Resident 2-CTA clusters of the pair kernel per device (the persistent grid
// must not exceed it), queried once.
int pair_clusters(bool tree) {
  static std::mutex mu;
  static int cache[64][2];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& row : cache) row[0] = row[1] = -1;
    init = true;
  }
  int& n = cache[dev][tree ? 1 : 0];
  if (n < 0) {
    auto kern = tree ? attn_mla_pair_kernel<true> : attn_mla_pair_kernel<false>;
    n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pr::kSmemBytes) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = pr::kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
  }
  return n;
}

}  // namespace

int mla_tc_split_granularity() { return kKeys; }

cudaError_t launch_attention_mla_tc(const mtp_attn_args& a, const AttnPlan& pl, unsigned* err, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  if (pl.split_len % kKeys) return cudaErrorInvalidValue;
  const int R = a.D + 1, rows = R * a.Hq;
  CUtensorMap tq, tkv;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kDQ, (cuuint64_t)a.B * rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kDQ * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kRows};
    if (!make_bf16_map(&tq, a.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDQ, (cuuint64_t)kBlock, (cuuint64_t)a.num_blocks};
    const cuuint64_t strides[2] = {(cuuint64_t)kDQ * 2, (cuuint64_t)kBlock * kDQ * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kBlock, 1};
    if (!make_bf16_map(&tkv, a.k_cache, 3, dims, strides, box)) return cudaErrorInvalidValue;
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
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.scale_log2 = a.sm_scale * kLog2e;
  const int row_blocks = (rows + kRows - 1) / kRows;
  // Row blocks pair up: the CTA-pair kernel; otherwise one CTA per row block.
  const bool paired = row_blocks % 2 == 0;
  const int C = paired ? 2 : 1;
  p.cluster = C;
  p.groups = row_blocks / C;
  const int n_items = pl.n_splits * a.B * p.groups;
  p.n_items = n_items;
  // CTA pairs are persistent: one pair per resident cluster slot (at most one
  // per item) walks its share of the order.
  int n_pairs = n_items;
  if (paired) {
    const int slots = pair_clusters(a.parents != nullptr);
    if (slots <= 0) return cudaErrorInvalidConfiguration;
    n_pairs = std::min(n_items, slots);
  }
  mla_schedule_kernel<<<1, 1024, 0, s>>>(a.ctx_lens, a.B, R, a.Hq, C, p.groups, pl.split_len, pl.n_splits,
                                         a.max_blocks * kBlock, (int32_t*)((char*)a.workspace + pl.ws_order));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int smem_bytes = paired ? pr::kSmemBytes : kSmemBytes;
  const bool tree = a.parents != nullptr;
  auto kern = paired ? (tree ? attn_mla_pair_kernel<true> : attn_mla_pair_kernel<false>)
                     : (tree ? attn_mla_tc_kernel<true> : attn_mla_tc_kernel<false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_pairs * C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tq, tkv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mtp
