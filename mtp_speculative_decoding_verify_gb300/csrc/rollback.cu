// KV-cache rollback after verification.
//
// "MTP in TensorRT-LLM", MTP Vanilla / MTP Eagle and the Fig. 4 workflow:
// once the accepted tokens are known, the keys/values of the discarded drafts
// are cleared from the KV cache (outside the engine forward). "Multi Token
// Prediction" note, rollback mechanism: the verified prefix stays as it is.
//
// The verify step wrote K/V into slots ctx .. ctx+D; the input token and the
// n accepted drafts keep theirs, so the sequence length becomes ctx + n + 1.
// Blocks that held verify slots but no kept slot return to the free list in
// request order, then block order. One CTA walks the batch in chunks of its
// thread count with a block-wide exclusive scan of the per-request counts.
//
// A request is rolled back whole or not at all: if the free list cannot take
// all of its freed blocks (counting every earlier request's blocks), its
// table row and length stay as they were and MTP_ERR_FREE_LIST is raised.
// The running count is monotone, so past the first request that does not fit
// only requests that free nothing are still rolled back; *free_count ends at
// the last block actually appended.
#include "common.cuh"
#include "kernels.h"

namespace mtp {

namespace {
constexpr int kThreads = 1024;
}

__global__ void __launch_bounds__(kThreads) kv_rollback_kernel(int32_t* __restrict__ block_table,
                                                               int32_t* __restrict__ seq_lens,
                                                               const int32_t* __restrict__ num_accepted,
                                                               int32_t* __restrict__ free_list,
                                                               int32_t* __restrict__ free_count, int B, int D,
                                                               int max_blocks, int capacity, unsigned* err) {
  __shared__ int s_warp[kThreads / kWarp];
  __shared__ int s_base;   // free-list position of the chunk's first block (all earlier requests counted)
  __shared__ int s_end;    // one past the last block appended
  const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
  if (tid == 0) s_base = s_end = *free_count;
  __syncthreads();
  for (int start = 0; start < B; start += kThreads) {
    const int b = start + tid;
    int first = 0, cnt = 0, kept = 0;
    if (b < B) {
      const int ctx = seq_lens[b];
      const int n = num_accepted[b];
      if (ctx < 0 || (ctx + D) / kBlock >= max_blocks) {
        raise_error(err, MTP_ERR_LENGTH);
        kept = -1;
      } else if (n < 0 || n > D) {
        raise_error(err, MTP_ERR_ACCEPTED);
        kept = -1;
      } else {
        kept = ctx + n + 1;
        first = (kept + kBlock - 1) / kBlock;
        const int last = (ctx + D) / kBlock;
        cnt = last >= first ? last - first + 1 : 0;
      }
    }
    // Block-wide exclusive scan of cnt.
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == kWarp - 1) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - cnt + (warp > 0 ? s_warp[warp - 1] : 0);
    const int total = s_warp[kWarp - 1];
    if (b < B && kept >= 0) {
      const int pos0 = s_base + excl;
      if (cnt == 0 || (pos0 >= 0 && (long long)pos0 + cnt <= (long long)capacity)) {
        int32_t* row = block_table + (int64_t)b * max_blocks;
        for (int i = 0; i < cnt; ++i) {
          free_list[pos0 + i] = row[first + i];
          row[first + i] = -1;
        }
        seq_lens[b] = kept;
        if (cnt > 0) atomicMax(&s_end, pos0 + cnt);
      } else {
        raise_error(err, MTP_ERR_FREE_LIST);   // left as it was: table row, length
      }
    }
    __syncthreads();
    if (tid == 0) s_base += total;
    __syncthreads();
  }
  if (tid == 0) *free_count = s_end;
}

cudaError_t launch_rollback(const mtp_rollback_args& a, unsigned* err, cudaStream_t s) {
  kv_rollback_kernel<<<1, kThreads, 0, s>>>(a.block_table, a.seq_lens, a.num_accepted, a.free_list, a.free_count,
                                            a.B, a.D, a.max_blocks, a.free_capacity, err);
  return cudaGetLastError();
}

}  // namespace mtp
