// Read-bandwidth probe: a measurement aid for the benchmark, not part of the
// verify path. It streams a buffer from device memory once, either with
// 16-byte loads folded into one XOR (so no load can be dropped) or with bulk
// copies into shared memory, which gives the read-only ceiling that the memory-bound kernels of the verify
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

// The same stream through the bulk-copy engine (the path the attention and
// LM-head kernels read through): one thread per CTA keeps kStages copies of
// kChunk bytes in flight into a shared-memory ring, each completing on its own
// mbarrier, and waits (time-limited) for a stage's previous copy before
// reusing it. Grid-stride over the chunks.
constexpr int kChunk = 32768;
constexpr int kStages = 6;
constexpr int kBulkSmem = kChunk * kStages;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n  .reg .pred p;\n  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n  selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 63u) == 63u) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > limit_ns) return false;
    }
  }
}

__global__ void __launch_bounds__(32) hbm_read_probe_bulk_kernel(const uint8_t* __restrict__ p, size_t bytes,
                                                                 uint32_t* __restrict__ sink, unsigned* err) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t bar[kStages];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kStages; ++s)
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar[s])) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const size_t n_chunks = (bytes + kChunk - 1) / kChunk;
  constexpr uint64_t kLimitNs = 2000000000ull;
  size_t j = 0;   // copies issued by this CTA
  bool ok = true;
  for (size_t c = blockIdx.x; c < n_chunks && ok; c += gridDim.x, ++j) {
    const int st = (int)(j % kStages);
    const uint32_t fill = (uint32_t)(j / kStages);
    if (fill > 0 && !bar_wait(&bar[st], (fill - 1) & 1u, kLimitNs)) {
      ok = false;
      break;
    }
    const uint32_t size = (uint32_t)min((size_t)kChunk, bytes - c * kChunk);   // a multiple of 16
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&bar[st])), "r"(size)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(ring + (size_t)st * kChunk)),
        "l"(p + c * kChunk), "r"(size), "r"(smem_addr(&bar[st]))
        : "memory");
  }
  // Every copy must land before the CTA exits: wait for the last fill of each stage.
  uint32_t acc = 0;
  for (size_t k = j > (size_t)kStages ? j - kStages : 0; k < j; ++k) {
    const int st = (int)(k % kStages);
    if (bar_wait(&bar[st], (uint32_t)(k / kStages) & 1u, kLimitNs)) acc ^= *reinterpret_cast<const uint32_t*>(ring + (size_t)st * kChunk);
    else ok = false;
  }
  if (!ok) raise_error(err, MTP_ERR_TIMEOUT);
  atomicXor(sink, acc);
}

}  // namespace
}  // namespace mtp

extern "C" int mtp_hbm_read_probe(const void* buf, size_t bytes, uint32_t* sink, int32_t ctas_per_sm,
                                  int32_t bulk, void* stream) {
  mtp::set_launch_count(0);
  if (!buf || !sink) return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: NULL buffer or sink");
  if (((uintptr_t)buf) % 16 || bytes % 16)
    return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: buffer and size must be multiples of 16 bytes");
  if (ctas_per_sm < 1 || ctas_per_sm > 4)
    return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: ctas_per_sm outside [1, 4]");
  if (bulk != 0 && bulk != 1) return mtp::set_error(MTP_INVALID_ARG, "mtp_hbm_read_probe: bulk must be 0 or 1");
  if (bytes == 0) return MTP_OK;
  unsigned* err = nullptr;
  int sm_count = 0;
  int rc = mtp::device_context(&err, &sm_count);
  if (rc != MTP_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (bulk) {
    e = cudaFuncSetAttribute(mtp::hbm_read_probe_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mtp::kBulkSmem);
    if (e != cudaSuccess) return mtp::set_cuda_error(e, "read probe shared memory");
    mtp::hbm_read_probe_bulk_kernel<<<sm_count, 32, mtp::kBulkSmem, s>>>(static_cast<const uint8_t*>(buf), bytes,
                                                                           sink, err);
  } else {
    mtp::hbm_read_probe_kernel<<<sm_count * ctas_per_sm, mtp::kThreads, 0, s>>>(static_cast<const uint4*>(buf),
                                                                                 bytes / 16, sink);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return mtp::set_cuda_error(e, "read probe launch");
  mtp::set_launch_count(1);
  return MTP_OK;
}
