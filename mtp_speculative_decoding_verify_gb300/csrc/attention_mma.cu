// Verify attention on tensor cores (bf16).
#include "common.cuh"
#include "kernels.h"

namespace mtp {

bool attention_mma_supported(const mtp_attn_args& a) { (void)a; return false; }
cudaError_t launch_attention_mma(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s) {
  (void)a; (void)p; (void)err; (void)s;
  return cudaErrorNotSupported;
}
cudaError_t launch_attention_mla(const mtp_attn_args& a, const AttnPlan& p, unsigned* err, cudaStream_t s) {
  (void)a; (void)p; (void)err; (void)s;
  return cudaErrorNotSupported;
}

}  // namespace mtp
