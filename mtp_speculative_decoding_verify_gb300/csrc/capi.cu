// C ABI of the verify-step library: host-side validation, workspace planning
// and kernel launches. See include/mtp_verify.h for the contract.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "../../include/mtp_verify.h"
#include "kernels.h"

namespace mtp {
unsigned long long current_context_id();
int lmhead_simt_slices(int V, int sm_count);
int lmhead_tc_slices(int V, int M, int sm_count);
bool lmhead_tc_supported(const mtp_lmhead_args& a);
size_t accept_decision_bytes();
cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned* err, cudaStream_t s);
size_t accept_race_part_bytes();
cudaError_t launch_rng_debug(uint64_t seed, uint32_t b, uint32_t j, uint32_t tag, uint32_t v0, int n,
                             uint32_t* word0, float* race_e, float* accept_u, cudaStream_t s);
}  // namespace mtp

namespace {

thread_local std::string g_last_error;
thread_local int g_launches = 0;

cudaError_t record(void* ev, cudaStream_t s) {
  return ev ? cudaEventRecord(static_cast<cudaEvent_t>(ev), s) : cudaSuccess;
}

// One 4-byte error word per device: kernels OR their range-check failures
// into it; mtp_sync_status() reads and clears it.
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
struct DeviceCtx {
  unsigned long long ctx_id = 0;   // context the entries below belong to (0: not set up)
  unsigned* err = nullptr;
  int sm_count = 0;
};
DeviceCtx g_dev[kMaxDevices];
std::mutex g_dev_mutex;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MTP_CUDA_ERROR, "%s: %s", what, cudaGetErrorString(e));
}

// Per-device context: the device address of the error word (host code may
// not use the symbol itself) and the SM count. Set up on the first call on a
// device, and again whenever the device's context is not the one the address
// came from (after cudaDeviceReset the module is loaded anew, at a new address).
int device_ctx(DeviceCtx** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MTP_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceCtx& c = g_dev[dev];
  const unsigned long long id = mtp::current_context_id();
  if (id == 0 || c.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);   // also makes the primary context current
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    e = cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    c.err = static_cast<unsigned*>(p);
    c.ctx_id = mtp::current_context_id();
  }
  *out = &c;
  return MTP_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// ------------------------------------------------------------- validation
int check_attn(const mtp_attn_args* a) {
  if (!a) return fail(MTP_INVALID_ARG, "mtp_verify_attention: args is NULL");
  if (a->B < 0) return fail(MTP_INVALID_ARG, "B = %d < 0", a->B);
  if (a->D < 0 || a->D > MTP_MAX_DRAFTS) return fail(MTP_INVALID_ARG, "D = %d outside [0, %d]", a->D, MTP_MAX_DRAFTS);
  if (a->block_size != MTP_BLOCK_SIZE) return fail(MTP_INVALID_ARG, "block_size = %d, must be 64", a->block_size);
  if (a->max_blocks <= 0 || a->num_blocks <= 0) return fail(MTP_INVALID_ARG, "max_blocks/num_blocks must be > 0");
  if (a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv) return fail(MTP_INVALID_ARG, "Hq %% Hkv != 0");
  if (a->dtype != MTP_F32 && a->dtype != MTP_BF16) return fail(MTP_INVALID_ARG, "dtype %d", a->dtype);
  if (!(a->sm_scale > 0.0f)) return fail(MTP_INVALID_ARG, "sm_scale must be > 0");
  if (a->B > 0 && (!a->q || !a->k_new || !a->k_cache || !a->block_table || !a->ctx_lens || !a->out))
    return fail(MTP_INVALID_ARG, "a required pointer is NULL");
  if (a->is_mla) {
    if (a->dtype != MTP_BF16) return fail(MTP_UNSUPPORTED, "MLA attention is provided for bf16 only");
    if (a->Hkv != 1 || a->d_qk != 576 || a->d_v != 512)
      return fail(MTP_UNSUPPORTED, "MLA needs Hkv = 1, d_qk = 576, d_v = 512");
    if (a->v_new || a->v_cache) return fail(MTP_INVALID_ARG, "MLA takes v_new = v_cache = NULL");
  } else {
    if (a->B > 0 && (!a->v_new || !a->v_cache)) return fail(MTP_INVALID_ARG, "v_new / v_cache is NULL");
    if (a->d_qk != a->d_v || (a->d_qk != 64 && a->d_qk != 128))
      return fail(MTP_UNSUPPORTED, "head dim must be 64 or 128 with d_qk == d_v");
  }
  return MTP_OK;
}

int check_lm(const mtp_lmhead_args* a) {
  if (!a) return fail(MTP_INVALID_ARG, "mtp_verify_logits_accept: args is NULL");
  if (a->B < 0) return fail(MTP_INVALID_ARG, "B = %d < 0", a->B);
  if (a->D < 0 || a->D > MTP_MAX_DRAFTS) return fail(MTP_INVALID_ARG, "D = %d outside [0, %d]", a->D, MTP_MAX_DRAFTS);
  if (a->H <= 0 || a->V <= 0) return fail(MTP_INVALID_ARG, "H and V must be > 0");
  if (a->dtype != MTP_F32 && a->dtype != MTP_BF16) return fail(MTP_INVALID_ARG, "dtype %d", a->dtype);
  if (a->dtype == MTP_F32 && a->H % 4) return fail(MTP_UNSUPPORTED, "fp32 LM head needs H %% 4 == 0");
  if (a->dtype == MTP_BF16 && a->H % 64) return fail(MTP_UNSUPPORTED, "bf16 LM head needs H %% 64 == 0");
  if ((long long)a->B * (a->D + 1) > (1 << 20)) return fail(MTP_UNSUPPORTED, "B*(D+1) > 2^20 rows");
  if (a->B > 0 && (!a->hidden || !a->lm_head || !a->tokens || !a->mode || !a->out_tokens || !a->num_accepted ||
                   !a->tie_flags))
    return fail(MTP_INVALID_ARG, "a required pointer is NULL");
  if (a->any_sampling && a->B > 0 && (!a->temperature || (a->D > 0 && !a->q_draft)))
    return fail(MTP_INVALID_ARG, "any_sampling = 1 needs temperature, and q_draft when D > 0");
  if (a->relaxed_topk < 0 || a->relaxed_topk > a->V)
    return fail(MTP_INVALID_ARG, "relaxed_topk = %d outside [0, V]", a->relaxed_topk);
  if (a->relaxed_topk > 0 && !(a->relaxed_delta >= 0.0f && a->relaxed_delta <= 1e30f))
    return fail(MTP_INVALID_ARG, "relaxed_delta must be finite and >= 0");
  return MTP_OK;
}

int check_rb(const mtp_rollback_args* a) {
  if (!a) return fail(MTP_INVALID_ARG, "kv_rollback: args is NULL");
  if (a->B < 0) return fail(MTP_INVALID_ARG, "B = %d < 0", a->B);
  if (a->D < 0 || a->D > MTP_MAX_DRAFTS) return fail(MTP_INVALID_ARG, "D = %d outside [0, %d]", a->D, MTP_MAX_DRAFTS);
  if (a->block_size != MTP_BLOCK_SIZE) return fail(MTP_INVALID_ARG, "block_size = %d, must be 64", a->block_size);
  if (a->max_blocks <= 0 || a->free_capacity < 0) return fail(MTP_INVALID_ARG, "max_blocks / free_capacity");
  if (!a->block_table || !a->seq_lens || !a->num_accepted || !a->free_list || !a->free_count)
    return fail(MTP_INVALID_ARG, "a required pointer is NULL");
  return MTP_OK;
}

}  // namespace

// --------------------------------------------------------------- planning
mtp::LmPlan mtp::plan_lmhead(const mtp_lmhead_args& a, int sm_count) {
  mtp::LmPlan p{};
  const int R = a.D + 1;
  p.M = a.B * R;
  p.tc = mtp::lmhead_tc_supported(a) ? 1 : 0;
  p.slices = p.tc ? mtp::lmhead_tc_slices(a.V, p.M, sm_count) : mtp::lmhead_simt_slices(a.V, sm_count);
  // race grid: about 8 CTAs per SM over the batch (requests that need no draw exit at once)
  p.race_slices = std::max(1, std::min(64, (8 * sm_count + a.B - 1) / std::max(a.B, 1)));
  p.race_slices = std::min(p.race_slices, std::max(1, a.V / 1024));
  size_t off = 0;
  const size_t part = align256((size_t)p.slices * p.M * 4);
  p.off_pmax = off; off += part;
  p.off_psum = off; off += part;
  p.off_pbest = off; off += part;
  p.off_pidx = off; off += part;
  p.off_ldraft = off; off += align256((size_t)p.M * 4);
  p.off_lse = off; off += align256((size_t)p.M * 4);
  p.off_amax = off; off += align256((size_t)p.M * 4);
  p.off_dec = off; off += align256((size_t)a.B * mtp::accept_decision_bytes());
  p.off_race = off; off += align256((size_t)a.B * p.race_slices * mtp::accept_race_part_bytes());
  p.off_count = off; off += align256((size_t)a.B * 4);
  p.off_logits = off;
  if (a.any_sampling) off += align256((size_t)p.M * a.V * 4);
  p.off_lpre = off;
  p.off_rcnt = off;
  if (a.relaxed_topk > 0) {
    off += align256((size_t)p.M * 4);
    p.off_rcnt = off;
    off += align256((size_t)3 * p.slices * p.M * 4);
  }
  p.ws_bytes = off;
  return p;
}

namespace mtp {
// Host-side validation and per-device context shared with the other entry points.
int check_lmhead_args(const mtp_lmhead_args* a) { return check_lm(a); }
int device_context(unsigned** err, int* sm_count) {
  DeviceCtx* c = nullptr;
  const int rc = device_ctx(&c);
  if (rc != MTP_OK) return rc;
  *err = c->err;
  *sm_count = c->sm_count;
  return MTP_OK;
}
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
int set_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
void set_launch_count(int n) { g_launches = n; }
}  // namespace mtp

extern "C" {

const char* mtp_last_error(void) { return g_last_error.c_str(); }

int mtp_abi_version(void) { return MTP_ABI_VERSION; }

int mtp_last_launch_count(void) { return g_launches; }

size_t mtp_abi_struct_size(int which) {
  switch (which) {
    case 0: return sizeof(mtp_attn_args);
    case 1: return sizeof(mtp_lmhead_args);
    case 2: return sizeof(mtp_rollback_args);
    case 3: return sizeof(mtp_draft_args);
    case 4: return sizeof(mtp_kv_compact_args);
    default: return 0;
  }
}

size_t mtp_attention_workspace_size(const mtp_attn_args* a) {
  if (check_attn(a) != MTP_OK) return 0;
  DeviceCtx* c = nullptr;
  if (device_ctx(&c) != MTP_OK) return 0;
  return std::max<size_t>(256, mtp::plan_attention(*a, c->sm_count).ws_bytes);
}

int mtp_verify_attention(const mtp_attn_args* a, void* stream) {
  int rc = check_attn(a);
  if (rc != MTP_OK) return rc;
  g_launches = 0;
  if (a->B == 0) return MTP_OK;
  DeviceCtx* c = nullptr;
  if ((rc = device_ctx(&c)) != MTP_OK) return rc;
  const mtp::AttnPlan p = mtp::plan_attention(*a, c->sm_count);
  if (p.ws_bytes > 0 && (!a->workspace || a->workspace_bytes < p.ws_bytes))
    return fail(MTP_INVALID_ARG, "workspace of %zu bytes needed, %zu given", p.ws_bytes, a->workspace_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = mtp::launch_kv_append(*a, c->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "kv append launch");
  if ((e = record(a->timing_events[0], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  if (mtp::attention_uses_mla_tc(*a)) e = mtp::launch_attention_mla(*a, p, c->err, s);
  else if (mtp::attention_uses_gqa_tc(*a)) e = mtp::launch_attention_gqa_tc(*a, p, c->err, s);
  else if (a->dtype == MTP_BF16 && mtp::attention_mma_supported(*a)) e = mtp::launch_attention_mma(*a, p, c->err, s);
  else e = mtp::launch_attention_simt(*a, p, c->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if ((e = record(a->timing_events[1], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  e = mtp::launch_attention_combine(*a, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "attention combine launch");
  // + the work-order kernel of every tensor-core attention path (MLA, GQA tcgen05, GQA mma.sync)
  g_launches = 2 + (p.n_splits > 1 ? 1 : 0) + (a->dtype == MTP_BF16 && mtp::attention_mma_supported(*a) ? 1 : 0);
  return MTP_OK;
}

size_t mtp_lmhead_workspace_size(const mtp_lmhead_args* a) {
  if (check_lm(a) != MTP_OK) return 0;
  DeviceCtx* c = nullptr;
  if (device_ctx(&c) != MTP_OK) return 0;
  return std::max<size_t>(256, mtp::plan_lmhead(*a, c->sm_count).ws_bytes);
}

int mtp_verify_logits_accept(const mtp_lmhead_args* a, void* stream) {
  int rc = check_lm(a);
  if (rc != MTP_OK) return rc;
  g_launches = 0;
  if (a->B == 0) return MTP_OK;
  DeviceCtx* c = nullptr;
  if ((rc = device_ctx(&c)) != MTP_OK) return rc;
  const mtp::LmPlan p = mtp::plan_lmhead(*a, c->sm_count);
  if (!a->workspace || a->workspace_bytes < p.ws_bytes)
    return fail(MTP_INVALID_ARG, "workspace of %zu bytes needed, %zu given", p.ws_bytes, a->workspace_bytes);
  if (((uintptr_t)a->workspace) % 256) return fail(MTP_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = mtp::launch_relaxed_prepass(*a, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "relaxed pre-pass launch");
  if ((e = record(a->timing_events[0], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  e = p.tc ? mtp::launch_lmhead_tc(*a, p, c->err, s) : mtp::launch_lmhead_simt(*a, p, c->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "LM head launch");
  if ((e = record(a->timing_events[1], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  if (a->q_ready_event && (e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(a->q_ready_event), 0)) != cudaSuccess)
    return cuda_fail(e, "cudaStreamWaitEvent(q_ready_event)");
  e = mtp::launch_accept(*a, p, c->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "accept launch");
  g_launches = 2 + (a->any_sampling ? 1 : 0) + (a->relaxed_topk > 0 ? 1 : 0);
  return MTP_OK;
}

int kv_rollback(const mtp_rollback_args* a, void* stream) {
  int rc = check_rb(a);
  if (rc != MTP_OK) return rc;
  g_launches = 0;
  if (a->B == 0) return MTP_OK;
  DeviceCtx* c = nullptr;
  if ((rc = device_ctx(&c)) != MTP_OK) return rc;
  cudaError_t e = mtp::launch_rollback(*a, c->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rollback launch");
  g_launches = 1;
  return MTP_OK;
}

int mtp_rng_debug(uint64_t seed, uint32_t b, uint32_t j, uint32_t tag, uint32_t v0, int32_t n, uint32_t* word0,
                  float* race_e, float* accept_u, void* stream) {
  if (n < 0) return fail(MTP_INVALID_ARG, "mtp_rng_debug: n = %d < 0", n);
  cudaError_t e = mtp::launch_rng_debug(seed, b, j, tag, v0, n, word0, race_e, accept_u,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rng debug launch");
  return MTP_OK;
}

int mtp_wait_selftest(uint64_t timeout_ns, void* stream) {
  if (timeout_ns < 1 || timeout_ns > 1000000000ull)
    return fail(MTP_INVALID_ARG, "mtp_wait_selftest: timeout %llu ns outside 1 .. 1e9", (unsigned long long)timeout_ns);
  DeviceCtx* c = nullptr;
  int rc = device_ctx(&c);
  if (rc != MTP_OK) return rc;
  cudaError_t e = mtp::launch_wait_selftest(timeout_ns, c->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait selftest launch");
  g_launches = 1;
  return MTP_OK;
}

int mtp_sync_status(void* stream) {
  DeviceCtx* c = nullptr;
  int rc = device_ctx(&c);
  if (rc != MTP_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, c->err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
  if (word == 0) return MTP_OK;
  e = cudaMemset(c->err, 0, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
  return fail(MTP_DEVICE_ERROR, "device range check failed: 0x%x%s%s%s%s%s%s%s%s", word,
              (word & MTP_ERR_BLOCK_ID) ? " block-id" : "", (word & MTP_ERR_TOKEN_ID) ? " token-id" : "",
              (word & MTP_ERR_LENGTH) ? " length" : "", (word & MTP_ERR_ACCEPTED) ? " num-accepted" : "",
              (word & MTP_ERR_FREE_LIST) ? " free-list" : "", (word & MTP_ERR_TIMEOUT) ? " timeout" : "",
              (word & MTP_ERR_MODE) ? " mode" : "", (word & MTP_ERR_TREE) ? " tree" : "");
}

}  // extern "C"
