// mtp_verify_logits_accept_noalloc: the LM-head + acceptance call for callers
// that cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer for the workspace: a
// plugin inside an inference engine that owns all device memory and hands
// plugins none, or a latency-critical loop where cudaMalloc's implicit
// device-wide synchronisation is not acceptable. This entry point takes the
// same arguments as mtp_verify_logits_accept but ignores `workspace` /
// `workspace_bytes`: its scratch lives in a fixed array in device memory that
// belongs to the library (kNoAllocScratchBytes; every GPU that loads the
// library holds it until the process exits). Inputs and outputs are still
// the caller's. Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mtp_verify.h"
#include "kernels.h"

namespace mtp {
unsigned long long current_context_id();
int check_lmhead_args(const mtp_lmhead_args* a);
int device_context(unsigned** err, int* sm_count);
int set_error(int code, const char* msg);
int set_cuda_error(cudaError_t e, const char* what);
void set_launch_count(int n);
}  // namespace mtp

namespace {

// 8 MiB of scratch: per-slice row statistics for up to a few thousand rows,
// plus full logit rows only when some request samples (M * V * 4 bytes).
constexpr size_t kNoAllocScratchBytes = MTP_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id = 0;   // context the address belongs to (0: not looked up yet)
  void* ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device. Host code must
// not use the symbol itself: on the host it names a stand-in, not device
// memory. Looked up with the device current, on the first call on that
// device and again whenever the device's context is not the one the address
// came from (a cudaDeviceReset loads the module anew, at a new address).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return mtp::set_error(MTP_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchSlot& slot = g_scratch[dev];
  const unsigned long long id = mtp::current_context_id();
  if (id == 0 || slot.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return mtp::set_cuda_error(e, "cudaGetSymbolAddress(no-alloc scratch)");
    slot.ptr = p;
    slot.ctx_id = mtp::current_context_id();
  }
  *out = slot.ptr;
  return MTP_OK;
}

}  // namespace

extern "C" size_t mtp_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int mtp_verify_logits_accept_noalloc(const mtp_lmhead_args* args, void* stream) {
  int rc = mtp::check_lmhead_args(args);
  if (rc != MTP_OK) return rc;
  mtp::set_launch_count(0);
  if (args->B == 0) return MTP_OK;
  unsigned* err = nullptr;
  int sm_count = 0;
  if ((rc = mtp::device_context(&err, &sm_count)) != MTP_OK) return rc;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != MTP_OK) return rc;
  mtp_lmhead_args a = *args;
  const mtp::LmPlan p = mtp::plan_lmhead(a, sm_count);
  if (p.ws_bytes > kNoAllocScratchBytes)
    return mtp::set_error(MTP_INVALID_ARG,
                          "mtp_verify_logits_accept_noalloc: this batch needs more scratch than the fixed "
                          "no-alloc array holds (see mtp_noalloc_scratch_bytes); use mtp_verify_logits_accept");
  a.workspace = scratch;
  a.workspace_bytes = kNoAllocScratchBytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = mtp::launch_relaxed_prepass(a, p, s);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "relaxed pre-pass launch");
  e = a.timing_events[0] ? cudaEventRecord(static_cast<cudaEvent_t>(a.timing_events[0]), s) : cudaSuccess;
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "cudaEventRecord");
  e = p.tc ? mtp::launch_lmhead_tc(a, p, err, s) : mtp::launch_lmhead_simt(a, p, err, s);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "LM head launch");
  e = a.timing_events[1] ? cudaEventRecord(static_cast<cudaEvent_t>(a.timing_events[1]), s) : cudaSuccess;
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "cudaEventRecord");
  e = a.q_ready_event ? cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(a.q_ready_event), 0) : cudaSuccess;
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "cudaStreamWaitEvent(q_ready_event)");
  e = mtp::launch_accept(a, p, err, s);
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "accept launch");
  mtp::set_launch_count(2 + (a.any_sampling ? 1 : 0) + (a.relaxed_topk > 0 ? 1 : 0));
  return MTP_OK;
}
