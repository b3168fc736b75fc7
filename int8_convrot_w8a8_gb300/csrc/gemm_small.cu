// Small-M int8 GEMM (M <= 64): a weight stream.
//
//   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]          (exact, int32)
//   Y[r, o] = bf16( fma(float(A[r,o]), s_x[r] * s_w[o], b[o]) )
//
// ("INT8 Convrot Safetensors", "Runtime activation quantization"; the
// gated-FFN pair sharing one packed activation follows gemma.cpp's W8A8
// report, "Implementation".)
//
// With a handful of rows every weight byte is used M times, so the layer is
// bound by reading the int8 weights once from HBM. Each CTA owns BNS output
// columns (BNS weight rows) of one linear and streams them, with the whole
// activation, through a TMA ring of 128-byte-wide K slices (128B swizzle).
// The ring is deep enough that typical K (<= 12 slices of 128) is requested
// in one go, so a CTA pays one memory round trip. A producer warp issues the
// copies; four consumer warps run mma.sync m16n8k32 s8 (native int32
// accumulation) on ldmatrix fragments and apply the fused epilogue. Waits are
// bounded and report CONVROT_ERR_TIMEOUT.
#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"
#include "tc_common.cuh"

namespace convrot {

namespace {

using namespace tc;

CONVROT_DEFINE_STATUS_WORD(status_word_small_local)

constexpr int SK = 128;          // K bytes per stage (one 128B swizzle atom per row)
constexpr int BNS = 32;          // weight rows per CTA
constexpr int MAX_STAGES = 12;
constexpr int CONSUMERS = 4;     // consumer warps: 8 output columns each
constexpr int THREADS_S = 32 * (CONSUMERS + 1);

struct SmallParams {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b[kMaxLinears];
  GemmOutputs outs;
  const float* sx;
  long long M;
  int K;
  int stages;
  int ktiles;
  long long spin_limit;
};

__device__ __forceinline__ void ldsm_x4s(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2s(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Byte offset of (row, 16-byte chunk) in a [rows][128 B] tile written by TMA
// with the 128B swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
  return static_cast<uint32_t>(row * SK + ((chunk ^ (row & 7)) << 4));
}

template <int MT, bool RAW>
__global__ void __launch_bounds__(THREADS_S) gemm_small_kernel(const __grid_constant__ SmallParams p) {
  constexpr int A_ROWS = 16 * MT;
  constexpr int A_BYTES = A_ROWS * SK;
  constexpr int B_BYTES = BNS * SK;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * STAGE_BYTES);
  uint64_t* empty = full + MAX_STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // which linear and which column block
  const int tile_n = blockIdx.x;
  int li = 0;
  while (li + 1 < p.outs.count && tile_n >= p.outs.o[li + 1].tile_begin) ++li;
  const GemmOut& out = p.outs.o[li];
  const int n0 = (tile_n - out.tile_begin) * BNS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CONSUMERS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == CONSUMERS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // The weights do not depend on the previous kernel of the stream (a
      // programmatic dependent launch: the rotate+quantize that writes the
      // codes): the first ring's weight tiles are requested before waiting
      // for it, the activation tiles after.
      const int first = p.ktiles < p.stages ? p.ktiles : p.stages;
      for (int kt = 0; kt < first; ++kt) {
        const uint32_t sa = sbase + kt * STAGE_BYTES;
        mbar_expect_tx(&full[kt], STAGE_BYTES);
        tma_load_2d(sa + A_BYTES, &p.tmap_b[li], kt * SK, n0, &full[kt]);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int kt = 0; kt < p.ktiles; ++kt) {
        const int s = kt % p.stages, round = kt / p.stages;
        const uint32_t sa = sbase + s * STAGE_BYTES;
        if (round > 0) {
          if (!mbar_wait_bounded(&empty[s], (round - 1) & 1, p.spin_limit)) {
            record_status(CONVROT_ERR_TIMEOUT);
            break;
          }
          mbar_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(sa + A_BYTES, &p.tmap_b[li], kt * SK, n0, &full[s]);
        }
        tma_load_2d(sa, &p.tmap_a, kt * SK, 0, &full[s]);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    // warp w: output columns n0 + 8w .. n0 + 8w + 7, all A_ROWS rows
    int acc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = 0;
    bool ok = true;
    for (int kt = 0; kt < p.ktiles; ++kt) {
      const int s = kt % p.stages, round = kt / p.stages;
      const bool got = ok && mbar_wait_bounded(&full[s], round & 1, p.spin_limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0 && ok) record_status(CONVROT_ERR_TIMEOUT);
        ok = false;
      }
      if (ok) {
        const uint32_t sa = sbase + s * STAGE_BYTES;
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < SK / 32; ++kk) {
          // B fragment: 8 columns (weight rows) x 32 k: matrices (rows, k 0-15) and (rows, k 16-31)
          uint32_t b0, b1;
          {
            const int j = (lane >> 3) & 1;
            const int row = warp * 8 + (lane & 7);
            ldsm_x2s(sb + sw_off(row, kk * 2 + j), b0, b1);
          }
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            uint32_t a[4];
            const int j = lane >> 3;
            const int row = i * 16 + (lane & 7) + 8 * (j & 1);
            ldsm_x4s(sa + sw_off(row, kk * 2 + (j >> 1)), a[0], a[1], a[2], a[3]);
            mma_s8_16832(acc[i], a, b0, b1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // ---- epilogue: fragment (g = lane/4, t = lane%4) holds rows g, g+8 and
    // columns 2t, 2t+1 of each 16x8 tile; the row scales come from the
    // previous kernel of the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int g = lane >> 2, t = lane & 3;
    const int c = n0 + warp * 8 + 2 * t;
    const int N = out.n;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const long long r = i * 16 + g + 8 * hr;
        if (r >= p.M || c >= N) continue;
        const int a0 = acc[i][2 * hr], a1 = acc[i][2 * hr + 1];
        if constexpr (RAW) {
          int* yp = static_cast<int*>(out.y) + r * out.ldy + c;
          if (c + 1 < N) {
            *reinterpret_cast<int2*>(yp) = make_int2(a0, a1);
          } else {
            yp[0] = a0;
          }
        } else {
          const float srow = p.sx[r];
          __nv_bfloat16* yp = static_cast<__nv_bfloat16*>(out.y) + r * out.ldy + c;
          const float bb0 = out.bias ? out.bias[c] : 0.0f;
          const float y0 = fmaf(static_cast<float>(a0), srow * out.sw[c], bb0);
          if (c + 1 < N) {
            const float bb1 = out.bias ? out.bias[c + 1] : 0.0f;
            const float y1 = fmaf(static_cast<float>(a1), srow * out.sw[c + 1], bb1);
            *reinterpret_cast<__nv_bfloat162*>(yp) = __floats2bfloat162_rn(y0, y1);
          } else {
            yp[0] = __float2bfloat16_rn(y0);
          }
        }
      }
    }
  }
}

bool make_map_u8(EncodeTiledFn enc, CUtensorMap* map, const void* base, long long rows, int K, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(SK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MT, bool RAW>
cudaError_t launch_small(EncodeTiledFn enc, const int8_t* Qx, const float* sx, long long M, int K, GemmOutputs outs,
                         cudaStream_t st) {
  SmallParams p;
  memset(&p, 0, sizeof(p));
  if (!make_map_u8(enc, &p.tmap_a, Qx, M, K, 16 * MT)) return cudaErrorInvalidValue;
  int nt = 0;
  for (int i = 0; i < outs.count; ++i) {
    outs.o[i].tile_begin = nt;
    nt += (outs.o[i].n + BNS - 1) / BNS;
    if (!make_map_u8(enc, &p.tmap_b[i], outs.o[i].qw, outs.o[i].n, K, BNS)) return cudaErrorInvalidValue;
  }
  p.outs = outs;
  p.sx = sx;
  p.M = M;
  p.K = K;
  p.ktiles = (K + SK - 1) / SK;
  p.stages = std::min(p.ktiles, MAX_STAGES);
  p.spin_limit = kDefaultSpinLimit;
  const int stage_bytes = (16 * MT + BNS) * SK;
  const int smem = 1024 + p.stages * stage_bytes + 2 * MAX_STAGES * 8;
  auto kern = gemm_small_kernel<MT, RAW>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  if (nt > 0x7fffffff) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nt);
  cfg.blockDim = dim3(THREADS_S);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int status_word_gemm_small() { return status_word_small_local(); }

bool gemm_small_supported(long long M, int K) { return M >= 1 && M <= 64 && K >= 16; }

cudaError_t gemm_small_launch(const int8_t* Qx, const float* sx, long long M, int K, const GemmOutputs& outs,
                              bool raw, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  if (M <= 16) return raw ? launch_small<1, true>(enc, Qx, sx, M, K, outs, st) : launch_small<1, false>(enc, Qx, sx, M, K, outs, st);
  if (M <= 32) return raw ? launch_small<2, true>(enc, Qx, sx, M, K, outs, st) : launch_small<2, false>(enc, Qx, sx, M, K, outs, st);
  return raw ? launch_small<4, true>(enc, Qx, sx, M, K, outs, st) : launch_small<4, false>(enc, Qx, sx, M, K, outs, st);
}

}  // namespace convrot
