// Read-bandwidth probe: a measurement aid for the benchmark, not part of the
// verify path. It streams a buffer from device memory once with 16-byte
// loads and folds every word into one XOR (so no load can be dropped), which
// gives the read-only ceiling that the memory-bound kernels of the verify
// step (KV-cache and LM-head weight streams, both read-only) are held
// against. A device-to-device copy moves each byte twice and turns the bus
// around between reads and writes, so a read stream can run faster than the
// copy rate.
#include <cuda_runtime.h>

#include "../../include/mtp_verify.h"
#include "common.cuh"

namespace mtp {
int device_context(unsigned** err, int* sm_count);
int set_error(int code, const char* msg);
int set_cuda_error(cudaError_t e, const char* what);
void set_launch_count(int n);

namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 8;   // loads in flight per thread

__global__ void __launch_bounds__(kThreads) hbm_read_probe_kernel(const uint4* __restrict__ p, size_t n,
                                                                  uint32_t* __restrict__ sink) {
  const size_t stride = (size_t)gridDim.x * kThreads;
  size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n; i += stride) {
    const uint4 v = __ldcs(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace
}  // namespace mtp

extern "C" int mtp_hbm_read_probe(const void* buf, size_t bytes, uint32_t* sink, int32_t ctas_per_sm,
                                  void* stream) {
  mtp::set_launch_count(0);
  if (!buf || !sink) return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: NULL buffer or sink");
  if (((uintptr_t)buf) % 16 || bytes % 16)
    return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: buffer and size must be multiples of 16 bytes");
  if (ctas_per_sm < 1 || ctas_per_sm > 4)
    return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: ctas_per_sm outside [1, 4]");
  if (bytes == 0) return MTP_OK;
  unsigned* err = nullptr;
  int sm_count = 0;
  int rc = mtp::device_context(&err, &sm_count);
  if (rc != MTP_OK) return rc;
  mtp::hbm_read_probe_kernel<<<sm_count * ctas_per_sm, mtp::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), bytes / 16, sink);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "read probe launch");
  mtp::set_launch_count(1);
  return MTP_OK;
}
