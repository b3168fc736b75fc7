// Rotation as a dense matmul -- placeholder until the kernel lands.
#include "common.cuh"

namespace convrot {

cudaError_t hmatmul_launch(const void*, long long, int, long long, int, int8_t*, float*, uint16_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace convrot
