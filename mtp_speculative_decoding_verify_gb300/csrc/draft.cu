// mtp_draft_argmax: one greedy draft step of MTP Eagle ("MTP in
// TensorRT-LLM on Blackwell", MTP Eagle; "MTP principles" §一: the MTP modules
// share the target's LM head and predict the drafts one after another).
//
// A draft step is the verify LM head with one row per request (R = 1, no
// drafts to check): the same tensor-core (or fp32 SIMT) GEMM streams W once
// with the fused (max, sum exp, argmax) epilogue, and the decide kernel
// merges the per-slice partials into each row's argmax and log-sum-exp.
#include <cuda_runtime.h>

#include "../../include/mtp_verify.h"
#include "kernels.h"

namespace mtp {
int device_context(unsigned** err, int* sm_count);
int set_error(int code, const char* msg);
int set_cuda_error(cudaError_t e, const char* what);
void set_launch_count(int n);
}  // namespace mtp

namespace {

int check_draft(const mtp_draft_args* a) {
  if (!a) return mtp::set_error(MTP_INVALID_ARG, "mtp_draft_argmax: args is NULL");
  if (a->B < 0) return mtp::set_error(MTP_INVALID_ARG, "mtp_draft_argmax: B < 0");
  if (a->H <= 0 || a->V <= 0) return mtp::set_error(MTP_INVALID_ARG, "mtp_draft_argmax: H and V must be > 0");
  if (a->dtype != MTP_F32 && a->dtype != MTP_BF16) return mtp::set_error(MTP_INVALID_ARG, "mtp_draft_argmax: dtype");
  if (a->dtype == MTP_F32 && a->H % 4) return mtp::set_error(MTP_UNSUPPORTED, "fp32 LM head needs H % 4 == 0");
  if (a->dtype == MTP_BF16 && a->H % 64) return mtp::set_error(MTP_UNSUPPORTED, "bf16 LM head needs H % 64 == 0");
  if (a->B > (1 << 20)) return mtp::set_error(MTP_UNSUPPORTED, "mtp_draft_argmax: B > 2^20 rows");
  if (a->B > 0 && (!a->hidden || !a->lm_head || !a->out_tokens))
    return mtp::set_error(MTP_INVALID_ARG, "mtp_draft_argmax: a required pointer is NULL");
  return MTP_OK;
}

// The verify LM head's arguments for R = 1 rows: no drafts, no mode array
// (every row greedy), no accept outputs.
mtp_lmhead_args as_lmhead(const mtp_draft_args& d) {
  mtp_lmhead_args a{};
  a.hidden = d.hidden;
  a.lm_head = d.lm_head;
  a.out_tokens = d.out_tokens;
  a.lse_out = d.lse_out;
  a.B = d.B;
  a.D = 0;
  a.H = d.H;
  a.V = d.V;
  a.dtype = d.dtype;
  a.workspace = d.workspace;
  a.workspace_bytes = d.workspace_bytes;
  a.timing_events[0] = d.timing_events[0];
  a.timing_events[1] = d.timing_events[1];
  return a;
}

cudaError_t record(void* ev, cudaStream_t s) {
  return ev ? cudaEventRecord(static_cast<cudaEvent_t>(ev), s) : cudaSuccess;
}

}  // namespace

extern "C" {

size_t mtp_draft_workspace_size(const mtp_draft_args* d) {
  if (check_draft(d) != MTP_OK) return 0;
  unsigned* err = nullptr;
  int sm_count = 0;
  if (mtp::device_context(&err, &sm_count) != MTP_OK) return 0;
  const size_t n = mtp::plan_lmhead(as_lmhead(*d), sm_count).ws_bytes;
  return n < 256 ? 256 : n;
}

int mtp_draft_argmax(const mtp_draft_args* d, void* stream) {
  int rc = check_draft(d);
  if (rc != MTP_OK) return rc;
  mtp::set_launch_count(0);
  if (d->B == 0) return MTP_OK;
  unsigned* err = nullptr;
  int sm_count = 0;
  if ((rc = mtp::device_context(&err, &sm_count)) != MTP_OK) return rc;
  const mtp_lmhead_args a = as_lmhead(*d);
  const mtp::LmPlan p = mtp::plan_lmhead(a, sm_count);
  if (!a.workspace || a.workspace_bytes < p.ws_bytes)
    return mtp::set_error(MTP_INVALID_ARG, "mtp_draft_argmax: workspace too small (see mtp_draft_workspace_size)");
  if (((uintptr_t)a.workspace) % 256) return mtp::set_error(MTP_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = record(a.timing_events[0], s);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "cudaEventRecord");
  e = p.tc ? mtp::launch_lmhead_tc(a, p, err, s) : mtp::launch_lmhead_simt(a, p, err, s);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "LM head launch");
  if ((e = record(a.timing_events[1], s)) != cudaSuccess) return mtp::set_cuda_error(e, "cudaEventRecord");
  e = mtp::launch_accept(a, p, err, s);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "argmax merge launch");
  mtp::set_launch_count(2);
  return MTP_OK;
}

}  // extern "C"
