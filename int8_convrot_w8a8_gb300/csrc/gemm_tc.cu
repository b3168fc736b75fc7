// Tensor-core (tcgen05) GEMM path -- placeholder until the kernel lands.
#include "common.cuh"
#include "gemm_common.cuh"

namespace convrot {

CONVROT_DEFINE_STATUS_WORD(status_word_gemm_tc)

bool gemm_tc_supported(long long, int) { return false; }

cudaError_t gemm_tc_launch(const uint16_t*, const float*, long long, int, const GemmOutputs&, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace convrot
