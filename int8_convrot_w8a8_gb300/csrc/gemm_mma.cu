// Int8 GEMM on the warp-level MMA path (mma.sync m16n8k32 s8 -> s32).
//
//   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]        (exact int32)
//   Y[r, o] = bf16( fma(float(A[r,o]), s_x[r] * s_w[o], b[o]) )
//
// ("INT8 Convrot Safetensors", "Runtime activation quantization": the int32
// accumulation and the reconstruction Y = A * s_x * s_w + b.)
//
// This path reads the int8 operands directly. It serves any shape with more
// than 64 rows for which no fp16 operand copies were provided (fewer rows go
// to the weight-stream kernel in gemm_small.cu). Operands are K-contiguous ("TN"); tiles
// of BK = 128 bytes of K are staged by cp.async in a multi-stage ring, rows
// XOR-swizzled by 16-byte chunk, and fed to the MMAs with ldmatrix.
#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"

namespace convrot {

CONVROT_DEFINE_STATUS_WORD(status_word_gemm_mma)

namespace {

constexpr int BK = 128;  // bytes of K per stage row

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of (row, 16-byte chunk) inside a [rows][128 B] stage tile.
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return static_cast<uint32_t>(row * BK + ((chunk ^ (row & 7)) << 4));
}

template <int BM, int BN, int WM, int WN, int STAGES, bool RAW>
__global__ void __launch_bounds__((BM / WM) * (BN / WN) * 32)
    gemm_mma_kernel(const int8_t* __restrict__ Qx, const float* __restrict__ sx, long long M, int K,
                    GemmOutputs outs) {
  constexpr int NWM = BM / WM, NWN = BN / WN;
  constexpr int THREADS = NWM * NWN * 32;
  constexpr int MT = WM / 16, NT = WN / 8;
  static_assert(NT % 2 == 0, "B fragments are loaded two n-tiles at a time");
  constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, STAGE_BYTES = A_BYTES + B_BYTES;

  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);

  // Which linear and which N tile this CTA owns.
  const int tile_n = blockIdx.y;
  int li = 0;
#pragma unroll 1
  while (li + 1 < outs.count && tile_n >= outs.o[li + 1].tile_begin) ++li;
  const GemmOut& out = outs.o[li];
  const int n0 = (tile_n - out.tile_begin) * BN;
  const int N = out.n;
  const int8_t* __restrict__ Qw = out.qw;
  const long long m0 = static_cast<long long>(blockIdx.x) * BM;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp / NWN, wn = warp % NWN;
  const int ktiles = (K + BK - 1) / BK;

  auto load_stage = [&](int stage, int kt) {
    const uint32_t sa = sbase + stage * STAGE_BYTES;
    const uint32_t sb = sa + A_BYTES;
    const int kbase = kt * BK;
    for (int c = tid; c < BM * (BK / 16); c += THREADS) {
      const int r = c / (BK / 16), ch = c % (BK / 16);
      const long long gr = m0 + r;
      const int k = kbase + ch * 16;
      const bool ok = gr < M && k < K;
      const int8_t* src = ok ? Qx + gr * K + k : Qx;
      cp_async_16(sa + tile_off(r, ch), src, ok ? 16 : 0);
    }
    for (int c = tid; c < BN * (BK / 16); c += THREADS) {
      const int r = c / (BK / 16), ch = c % (BK / 16);
      const int gn = n0 + r;
      const int k = kbase + ch * 16;
      const bool ok = gn < N && k < K;
      const int8_t* src = ok ? Qw + static_cast<long long>(gn) * K + k : Qw;
      cp_async_16(sb + tile_off(r, ch), src, ok ? 16 : 0);
    }
  };

  int acc[MT][NT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ktiles) load_stage(s, s);
    cp_async_commit();
  }

#pragma unroll 1
  for (int kt = 0; kt < ktiles; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const int nk = kt + STAGES - 1;
    if (nk < ktiles) load_stage(nk % STAGES, nk);
    cp_async_commit();

    const uint32_t sa = sbase + (kt % STAGES) * STAGE_BYTES;
    const uint32_t sb = sa + A_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 32; ++kk) {
      uint32_t af[MT][4];
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const int j = lane >> 3;
        const int row = wm * WM + i * 16 + (lane & 7) + 8 * (j & 1);
        const int chunk = kk * 2 + (j >> 1);
        ldsm_x4(sa + tile_off(row, chunk), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
      uint32_t bf[NT][2];
#pragma unroll
      for (int jj = 0; jj < NT; jj += 2) {
        const int j = lane >> 3;
        const int row = wn * WN + jj * 8 + (lane & 7) + 8 * (j >> 1);
        const int chunk = kk * 2 + (j & 1);
        ldsm_x4(sb + tile_off(row, chunk), bf[jj][0], bf[jj][1], bf[jj + 1][0], bf[jj + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
    }
  }
  cp_async_wait<0>();

  // ---- epilogue: fragment (g = lane/4, t = lane%4): rows g and g+8 of the
  // 16x8 tile, columns 2t and 2t+1.
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < MT; ++i) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const long long r = m0 + wm * WM + i * 16 + g + 8 * hr;
      if (r >= M) continue;
      const float srow = RAW ? 0.0f : sx[r];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = n0 + wn * WN + j * 8 + 2 * t;
        if (c >= N) continue;
        const int a0 = acc[i][j][2 * hr], a1 = acc[i][j][2 * hr + 1];
        if constexpr (RAW) {
          int* yp = static_cast<int*>(out.y) + r * out.ldy + c;
          if (c + 1 < N) {
            *reinterpret_cast<int2*>(yp) = make_int2(a0, a1);
          } else {
            yp[0] = a0;
          }
        } else {
          __nv_bfloat16* yp = static_cast<__nv_bfloat16*>(out.y) + r * out.ldy + c;
          const float b0 = out.bias ? out.bias[c] : 0.0f;
          const float y0 = fmaf(static_cast<float>(a0), srow * out.sw[c], b0);
          if (c + 1 < N) {
            const float b1 = out.bias ? out.bias[c + 1] : 0.0f;
            const float y1 = fmaf(static_cast<float>(a1), srow * out.sw[c + 1], b1);
            *reinterpret_cast<__nv_bfloat162*>(yp) = __floats2bfloat162_rn(y0, y1);
          } else {
            yp[0] = __float2bfloat16_rn(y0);
          }
        }
      }
    }
  }
}

template <int BM, int BN, int WM, int WN, int STAGES, bool RAW>
cudaError_t launch_cfg(const int8_t* Qx, const float* sx, long long M, int K, GemmOutputs outs, cudaStream_t st) {
  constexpr int THREADS = (BM / WM) * (BN / WN) * 32;
  constexpr int SMEM = STAGES * (BM + BN) * BK;
  int tiles_n = 0;
  for (int i = 0; i < outs.count; ++i) {
    outs.o[i].tile_begin = tiles_n;
    tiles_n += (outs.o[i].n + BN - 1) / BN;
  }
  auto kern = gemm_mma_kernel<BM, BN, WM, WN, STAGES, RAW>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), SMEM);
  if (e != cudaSuccess) return e;
  const long long tiles_m = (M + BM - 1) / BM;
  if (tiles_m > 0x7fffffffLL || tiles_n > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(tiles_m), static_cast<unsigned>(tiles_n));
  kern<<<grid, THREADS, SMEM, st>>>(Qx, sx, M, K, outs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_mma_launch(const int8_t* Qx, const float* sx, long long M, int K, const GemmOutputs& outs,
                            bool raw, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  return raw ? launch_cfg<128, 128, 64, 32, 3, true>(Qx, sx, M, K, outs, st)
             : launch_cfg<128, 128, 64, 32, 3, false>(Qx, sx, M, K, outs, st);
}

}  // namespace convrot
