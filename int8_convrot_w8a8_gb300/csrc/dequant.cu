// The reconstruction of "INT8 Convrot Safetensors" ("Runtime activation
// quantization": Y[r, o] ~= A[r, o] * s_x[r] * s_w[o] + b[o]) as a kernel of
// its own, for int32 accumulators that arrive from elsewhere: the sum of the
// partial products of a row-parallel (K-sharded) linear. Same expression and
// rounding as the GEMM epilogues, fmaf(float(A), s_x * s_w, b) rounded once
// to bf16, so Y is bit-identical to the fused path's.
#include <algorithm>

#include "common.cuh"

namespace convrot {

constexpr int kDqThreads = 128;  // threads of a block, one block of 8 columns each
constexpr int kDqRows = 4;       // rows a thread has in flight

// A thread owns 8 consecutive columns (their scales and biases stay in
// registers) and walks the rows of its block's row set, kDqRows at a time:
// two 16-byte int32 loads per row, all issued before the first is used, then
// one 16-byte bf16 store per row. A ragged last column block takes the
// element-wise branch; rows past M are skipped.
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const int32_t* __restrict__ A, long long M, int N,
                                                              long long lda, const float* __restrict__ sx,
                                                              const float* __restrict__ sw,
                                                              const float* __restrict__ bias,
                                                              __nv_bfloat16* __restrict__ Y, long long ldy) {
  const int c0 = (blockIdx.x * kDqThreads + threadIdx.x) * 8;
  if (c0 >= N) return;
  const long long r_step = static_cast<long long>(gridDim.y) * kDqRows;
  if (c0 + 8 <= N) {
    float w[8], b[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      w[e] = sw[c0 + e];
      b[e] = bias ? bias[c0 + e] : 0.0f;
    }
    for (long long r0 = static_cast<long long>(blockIdx.y) * kDqRows; r0 < M; r0 += r_step) {
      int4 a[kDqRows][2];
      float s[kDqRows];
#pragma unroll
      for (int j = 0; j < kDqRows; ++j) {
        const long long r = r0 + j < M ? r0 + j : M - 1;  // past M: a valid row, not stored
        const int4* p = reinterpret_cast<const int4*>(A + r * lda + c0);
        a[j][0] = __ldg(p);
        a[j][1] = __ldg(p + 1);
        s[j] = __ldg(sx + r);
      }
#pragma unroll
      for (int j = 0; j < kDqRows; ++j) {
        if (r0 + j >= M) break;
        const int av[8] = {a[j][0].x, a[j][0].y, a[j][0].z, a[j][0].w, a[j][1].x, a[j][1].y, a[j][1].z, a[j][1].w};
        __align__(16) __nv_bfloat16 out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = __float2bfloat16_rn(fmaf(static_cast<float>(av[e]), s[j] * w[e], b[e]));
        *reinterpret_cast<int4*>(Y + (r0 + j) * ldy + c0) = *reinterpret_cast<const int4*>(out);
      }
    }
  } else {
    for (long long r0 = static_cast<long long>(blockIdx.y) * kDqRows; r0 < M; r0 += r_step)
      for (long long r = r0; r < r0 + kDqRows && r < M; ++r) {
        const float s = sx[r];
        for (int e = 0; c0 + e < N; ++e)
          Y[r * ldy + c0 + e] =
              __float2bfloat16_rn(fmaf(static_cast<float>(A[r * lda + c0 + e]), s * sw[c0 + e], bias ? bias[c0 + e] : 0.0f));
      }
  }
}

cudaError_t dequant_launch(const int32_t* A, long long M, int N, long long lda, const float* sx, const float* sw,
                           const float* bias, uint16_t* Y, long long ldy, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const int cb = (N + 7) / 8;
  const unsigned gx = static_cast<unsigned>((cb + kDqThreads - 1) / kDqThreads);
  // enough resident blocks to keep HBM busy (16 per SM), no more row sets
  // than row groups
  const long long row_groups = (M + kDqRows - 1) / kDqRows;
  const long long want = (16LL * device_sm_count() + gx - 1) / gx;
  const unsigned gy = static_cast<unsigned>(std::min<long long>({row_groups, want, 65535LL}));
  dequant_kernel<<<dim3(gx, gy), kDqThreads, 0, st>>>(A, M, N, lda, sx, sw, bias,
                                                     reinterpret_cast<__nv_bfloat16*>(Y), ldy);
  return cudaGetLastError();
}

}  // namespace convrot
