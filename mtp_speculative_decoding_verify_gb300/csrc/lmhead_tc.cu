// LM head on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
#include "common.cuh"
#include "kernels.h"

namespace mtp {

bool lmhead_tc_supported(const mtp_lmhead_args& a) { (void)a; return false; }
int lmhead_tc_slices(int V, int M, int sm_count) { (void)V; (void)M; return sm_count; }
cudaError_t launch_lmhead_tc(const mtp_lmhead_args& a, const LmPlan& p, unsigned* err, cudaStream_t s) {
  (void)a; (void)p; (void)err; (void)s;
  return cudaErrorNotSupported;
}

}  // namespace mtp
