// mtp_tree_kv_compact: after a tree verify, move the accepted path's K/V into
// contiguous slots ("MTP in TensorRT-LLM on Blackwell", future work: tree
// speculative sampling, with the rollback of the MTP Vanilla / Eagle
// sections: only the accepted tokens keep their K/V).
//
// The verify call put node k's K/V at slot ctx + k. The kept sequence is the
// input token and the accepted path u_0 = 0, u_1 .. u_n, so slot ctx + u_i
// moves to slot ctx + i for i = 1 .. n. Path nodes increase (u_i >= i), so in
// increasing i a move never overwrites a slot that a later move still reads;
// one CTA per request does the moves in that order, its threads copying one
// token's K (and V) row together. kv_rollback then trims and frees blocks.
#include <cuda_runtime.h>

#include "../../include/mtp_verify.h"
#include "common.cuh"
#include "kernels.h"

namespace mtp {
int device_context(unsigned** err, int* sm_count);
int set_error(int code, const char* msg);
int set_cuda_error(cudaError_t e, const char* what);
void set_launch_count(int n);
}  // namespace mtp

namespace {

using mtp::kBlock;
using mtp::raise_error;

constexpr int kThreads = 128;

// Copy `bytes` (a multiple of 2) from src to dst with the widest aligned access.
__device__ __forceinline__ void copy_row(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src, int bytes) {
  if (bytes % 16 == 0 && (((uintptr_t)dst | (uintptr_t)src) & 15) == 0) {
    for (int i = threadIdx.x; i < bytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
  } else if (bytes % 4 == 0 && (((uintptr_t)dst | (uintptr_t)src) & 3) == 0) {
    for (int i = threadIdx.x; i < bytes / 4; i += kThreads)
      reinterpret_cast<uint32_t*>(dst)[i] = reinterpret_cast<const uint32_t*>(src)[i];
  } else {
    for (int i = threadIdx.x; i < bytes / 2; i += kThreads)
      reinterpret_cast<uint16_t*>(dst)[i] = reinterpret_cast<const uint16_t*>(src)[i];
  }
}

__global__ void __launch_bounds__(kThreads) tree_kv_compact_kernel(
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ ctx_lens, const int32_t* __restrict__ accepted_nodes,
    const int32_t* __restrict__ num_accepted, int D, int max_blocks, int num_blocks, int k_row_bytes,
    int v_row_bytes, unsigned* err) {
  const int b = blockIdx.x;
  const int R = D + 1;
  const int ctx = ctx_lens[b];
  const int n = num_accepted[b];
  // Every check below reads the same values in every thread, so an early
  // return leaves the whole CTA.
  if (n < 0 || n > D) {
    if (threadIdx.x == 0) raise_error(err, MTP_ERR_ACCEPTED);
    return;
  }
  if (ctx < 0 || (ctx + D) / kBlock >= max_blocks) {
    if (threadIdx.x == 0) raise_error(err, MTP_ERR_LENGTH);
    return;
  }
  const int32_t* path = accepted_nodes + (int64_t)b * R;
  bool ok = path[0] == 0;
  for (int i = 1; i <= n; ++i) ok = ok && path[i] > path[i - 1] && path[i] < R;
  if (!ok) {
    if (threadIdx.x == 0) raise_error(err, MTP_ERR_TREE);
    return;
  }
  const int32_t* tbl = block_table + (int64_t)b * max_blocks;
  for (int i = 1; i <= n; ++i) {
    const int src = path[i];
    if (src == i) continue;   // uniform: every thread skips
    const int ss = ctx + src, ds = ctx + i;
    const int sb = tbl[ss / kBlock], db = tbl[ds / kBlock];
    if (sb < 0 || sb >= num_blocks || db < 0 || db >= num_blocks) {
      if (threadIdx.x == 0) raise_error(err, MTP_ERR_BLOCK_ID);
      return;
    }
    const int64_t s_slot = (int64_t)sb * kBlock + ss % kBlock, d_slot = (int64_t)db * kBlock + ds % kBlock;
    copy_row(k_cache + d_slot * k_row_bytes, k_cache + s_slot * k_row_bytes, k_row_bytes);
    if (v_cache) copy_row(v_cache + d_slot * v_row_bytes, v_cache + s_slot * v_row_bytes, v_row_bytes);
    __syncthreads();   // this move has landed before a later move reads its source
  }
}

int check_compact(const mtp_kv_compact_args* a) {
  if (!a) return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: args is NULL");
  if (a->B < 0) return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: B < 0");
  if (a->D < 0 || a->D > MTP_MAX_DRAFTS) return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: D out of range");
  if (a->block_size != MTP_BLOCK_SIZE) return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: block_size must be 64");
  if (a->Hkv <= 0 || a->d_qk <= 0 || a->d_v <= 0 || a->max_blocks <= 0 || a->num_blocks <= 0)
    return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: sizes must be > 0");
  if (a->dtype != MTP_F32 && a->dtype != MTP_BF16) return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: dtype");
  if (a->is_mla && (a->Hkv != 1 || a->v_cache))
    return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: MLA takes Hkv = 1 and v_cache = NULL");
  if (a->B > 0 && (!a->k_cache || (!a->is_mla && !a->v_cache) || !a->block_table || !a->ctx_lens ||
                   !a->accepted_nodes || !a->num_accepted))
    return mtp::set_error(MTP_INVALID_ARG, "mtp_tree_kv_compact: a required pointer is NULL");
  return MTP_OK;
}

}  // namespace

extern "C" int mtp_tree_kv_compact(const mtp_kv_compact_args* a, void* stream) {
  int rc = check_compact(a);
  if (rc != MTP_OK) return rc;
  mtp::set_launch_count(0);
  if (a->B == 0) return MTP_OK;
  unsigned* err = nullptr;
  int sm_count = 0;
  if ((rc = mtp::device_context(&err, &sm_count)) != MTP_OK) return rc;
  const int elem = a->dtype == MTP_BF16 ? 2 : 4;
  tree_kv_compact_kernel<<<a->B, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(a->k_cache), static_cast<uint8_t*>(a->v_cache), a->block_table, a->ctx_lens,
      a->accepted_nodes, a->num_accepted, a->D, a->max_blocks, a->num_blocks, a->Hkv * a->d_qk * elem,
      a->Hkv * a->d_v * elem, err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "tree KV compaction launch");
  mtp::set_launch_count(1);
  return MTP_OK;
}
