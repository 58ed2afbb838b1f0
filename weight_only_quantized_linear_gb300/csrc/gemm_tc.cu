// gemm_tc.cu -- large-M group-wise 4-bit linear on the tcgen05 tensor cores.
#include "common.cuh"
#include "launch.h"

namespace wq {

bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, int32_t group) {
  (void)M; (void)N; (void)K; (void)group;
  return false;
}

cudaError_t launch_gemm_tc(const GemmTcParams& p, int num_sms, cudaStream_t stream) {
  (void)p; (void)num_sms; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace wq
