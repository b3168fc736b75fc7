// The reconstruction of "INT8 Convrot Safetensors" ("Runtime activation
// quantization": Y[r, o] ~= A[r, o] * s_x[r] * s_w[o] + b[o]) as a kernel of
// its own, for int32 accumulators that arrive from elsewhere: the sum of the
// partial products of a row-parallel (K-sharded) linear. Same expression and
// rounding as the GEMM epilogues, fmaf(float(A), s_x * s_w, b) rounded once
// to bf16, so Y is bit-identical to the fused path's.
#include "common.cuh"

namespace convrot {

// Eight outputs per thread: two 16-byte int32 loads, one 16-byte bf16 store
// (columns past N and rows past M are skipped; a ragged tail column block
// takes the element-wise branch).
__global__ void __launch_bounds__(256) dequant_kernel(const int32_t* __restrict__ A, long long M, int N,
                                                       long long lda, const float* __restrict__ sx,
                                                       const float* __restrict__ sw, const float* __restrict__ bias,
                                                       __nv_bfloat16* __restrict__ Y, long long ldy) {
  const int cb = (N + 7) / 8;  // column blocks of 8
  const long long total = M * cb;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / cb;
    const int c0 = static_cast<int>(i - r * cb) * 8;
    const float s = sx[r];
    const int32_t* a = A + r * lda + c0;
    __nv_bfloat16* y = Y + r * ldy + c0;
    if (c0 + 8 <= N) {
      const int4 a0 = *reinterpret_cast<const int4*>(a);
      const int4 a1 = *reinterpret_cast<const int4*>(a + 4);
      const int av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      __align__(16) __nv_bfloat16 out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        out[e] = __float2bfloat16_rn(fmaf(static_cast<float>(av[e]), s * sw[c0 + e], bias ? bias[c0 + e] : 0.0f));
      *reinterpret_cast<int4*>(y) = *reinterpret_cast<const int4*>(out);
    } else {
      for (int e = 0; c0 + e < N; ++e)
        y[e] = __float2bfloat16_rn(fmaf(static_cast<float>(a[e]), s * sw[c0 + e], bias ? bias[c0 + e] : 0.0f));
    }
  }
}

cudaError_t dequant_launch(const int32_t* A, long long M, int N, long long lda, const float* sx, const float* sw,
                           const float* bias, uint16_t* Y, long long ldy, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const long long total = M * ((N + 7) / 8);
  const long long want = (total + 255) / 256;
  const long long cap = 8LL * device_sm_count();  // enough resident blocks to stream at HBM speed
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  dequant_kernel<<<grid, 256, 0, st>>>(A, M, N, lda, sx, sw, bias, reinterpret_cast<__nv_bfloat16*>(Y), ldy);
  return cudaGetLastError();
}

}  // namespace convrot
