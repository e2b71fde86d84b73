// Internal launchers of the verify-step kernels (host side). Not part of the
// C ABI; capi.cu validates arguments and calls these.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mtp_verify.h"

namespace mtp {

// ---------------------------------------------------------------- attention
struct AttnPlan {
  int rows_per_kv;     // query rows sharing one KV head: (Hq/Hkv) * R
  int n_splits;        // KV splits per (request, KV head); 1 = no combine pass
  int split_len;       // keys per split (multiple of 64)
  size_t ws_partial_o; // byte offset of the split partial outputs in the workspace
  size_t ws_partial_lse;
  size_t ws_order;     // tensor-core MLA / GQA paths: work-item order (int32 per item)
  size_t ws_bytes;
  int sm_count;        // SMs of the device the plan is for
};

AttnPlan plan_attention(const mtp_attn_args& a, int sm_count);
cudaError_t launch_kv_append(const mtp_attn_args& a, unsigned* err, cudaStream_t s);
cudaError_t launch_attention_simt(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_attention_mma(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_attention_mla(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_attention_mla_tc(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s);
bool attention_mma_supported(const mtp_attn_args& a);   // bf16 GQA/MHA (d 64, 128) or MLA on tensor cores
bool attention_uses_mla_tc(const mtp_attn_args& a);
// bf16 GQA/MHA, head dim 128, 49..64 query rows per KV head: tcgen05 kernel
bool attention_uses_gqa_tc(const mtp_attn_args& a);
int attention_mma_row_tiles(const mtp_attn_args& a);      // CTAs per (split, request, KV head) of the mma.sync GQA kernel
cudaError_t launch_attention_gqa_tc(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_attention_combine(const mtp_attn_args& a, const AttnPlan& p, cudaStream_t s);

// ------------------------------------------------------------------ LM head
// Workspace of mtp_verify_logits_accept, all offsets in bytes.
struct LmPlan {
  int M;               // B * R rows
  int slices;          // vocab slices (one per LM-head CTA), partials per row
  int race_slices;     // vocab slices per sampling request in the race kernel
  int tc;              // 1: tcgen05 kernel, 0: SIMT kernel
  size_t off_pmax, off_psum, off_pbest, off_pidx;  // [slices][M]
  size_t off_ldraft;                               // [M] float
  size_t off_lse, off_amax;                        // [M]
  size_t off_dec;                                  // [B] int4 decision records
  size_t off_race;                                 // [B][race_slices] race partials (2 x Race)
  size_t off_count;                                // [B] int arrival counters
  size_t off_logits;                               // [M][V] float, sampling rows only
  size_t off_lpre;                                 // [M] float: draft logit of relaxed rows (pre-pass)
  size_t off_rcnt;                                 // [3][slices][M] int: relaxed rank counts per slice
  size_t ws_bytes;
};

LmPlan plan_lmhead(const mtp_lmhead_args& a, int sm_count);
cudaError_t launch_lmhead_simt(const mtp_lmhead_args& a, const LmPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_lmhead_tc(const mtp_lmhead_args& a, const LmPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_accept(const mtp_lmhead_args& a, const LmPlan& p, unsigned* err, cudaStream_t s);
cudaError_t launch_relaxed_prepass(const mtp_lmhead_args& a, const LmPlan& p, cudaStream_t s);

// ----------------------------------------------------------------- rollback
cudaError_t launch_rollback(const mtp_rollback_args& a, unsigned* err, cudaStream_t s);

}  // namespace mtp
