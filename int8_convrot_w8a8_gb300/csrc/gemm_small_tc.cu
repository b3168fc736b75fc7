// Small-M int8 GEMM (M <= 64) on the tcgen05 tensor cores: a weight stream.
//
//   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]          (exact, int32)
//   Y[r, o] = bf16( fma(float(A[r,o]), s_x[r] * s_w[o], b[o]) )
//
// ("INT8 Convrot Safetensors", "Runtime activation quantization"; the
// gated-FFN pair sharing one packed activation follows gemma.cpp's W8A8
// report, "Implementation".)
//
// With a handful of activation rows every weight byte is used M times, so the
// layer is bound by reading the int8 weights once from HBM. The roles of the
// operands are swapped: each CTA computes D = W_tile X^T, 128 weight rows
// (the MMA's M) by the NA activation rows (its N, M rounded up to 16), over
// the whole K, so no MMA work is spent on padding rows of a 128-row tile.
//
// sm_103a has no integer tcgen05 MMA and the legacy integer mma.sync runs
// an order of magnitude below the fp16 tensor rate, so the int8 tiles are
// widened to fp16 in shared memory (every integer in [-127, 127] is exact)
// and multiplied with kind::f16 into fp32 tensor memory. The weights still
// stream from HBM as int8, one byte per weight.
//
// Per K tile of 128 (one 128-byte row per operand row):
//   warp 0      TMA producer: int8 weight tile (128 x 128 B) and int8
//               activation tile (NA x 128 B), 128-byte swizzle, into a deep
//               ring; the fp16 tiles have a ring of their own.
//   warps 2..9  converters: each thread widens half a weight row (64 K
//               values, one fp16 atom row) and a share of the activation
//               rows into K-major 128-byte-swizzled fp16 atoms, the layout
//               the MMA descriptors describe.
//   warp 1      TMEM allocation and the MMA issuer: eight M = 128, N = NA,
//               K = 16 MMAs per tile. Partial sums stay exact while a chunk
//               spans at most 1024 of K (127 * 127 * 1024 < 2^24), so chunk
//               c accumulates into its own NA columns of tensor memory.
// After the last tile warps 2..9 read every chunk (tcgen05.ld; two warps per
// lane quadrant, half of the columns each), sum the chunks in int32 and
// apply the scale, bias and bf16 epilogue. Every wait is
// bounded and reports CONVROT_ERR_TIMEOUT.
#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"
#include "tc_common.cuh"

namespace convrot {

namespace {

using namespace tc;

CONVROT_DEFINE_STATUS_WORD(status_word_small_tc_local)

constexpr int KT = 128;             // K values per tile (one 128-byte int8 row)
constexpr int WROWS = 128;          // weight rows per CTA (the MMA's M)
constexpr int KCHUNK_TILES = 8;     // tiles per exact fp32 chunk (1024 of K)
constexpr int CONV_WARPS = 8;      // converter / epilogue warps
constexpr int THREADS_T = 32 * (2 + CONV_WARPS);
constexpr int MAX_STAGES8 = 12;     // int8 ring
constexpr int MAX_STAGES16 = 4;     // fp16 ring

template <int NA>
struct SCfg {
  static_assert(NA % 16 == 0 && NA >= 16 && NA <= 64, "activation rows padded to 16..64");
  static constexpr int W8 = WROWS * KT;                 // int8 weight tile
  static constexpr int X8 = ((NA * KT + 1023) / 1024) * 1024;
  static constexpr int STAGE8 = W8 + X8;                // a multiple of 1024
  static constexpr int W16 = 2 * WROWS * 128;           // two fp16 atoms of 64 K values
  static constexpr int X16 = 2 * NA * 128;
  static constexpr int STAGE16 = W16 + X16;             // a multiple of 1024
  static constexpr uint32_t IDESC = idesc_f16(WROWS, NA, false);
};

struct SmallTcParams {
  CUtensorMap tmap_x;
  CUtensorMap tmap_w[kMaxLinears];
  GemmOutputs outs;
  const float* sx;
  long long M;
  int K;
  int ktiles;
  int stages;      // int8 ring depth
  int stages16;    // fp16 ring depth
  uint32_t tmem_cols;
  long long spin_limit;
};

// int8 bytes b0..b3 of w -> fp16 pairs (b0, b1), (b2, b3): the bits 0x64uu
// with u = b + 128 are the fp16 value 1024 + u, so subtracting 1152 leaves b.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& h01, uint32_t& h23) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 off = __halves2half2(__float2half(1152.0f), __float2half(1152.0f));
  const __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), off);
  const __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), off);
  h01 = *reinterpret_cast<const uint32_t*>(&ha);
  h23 = *reinterpret_cast<const uint32_t*>(&hb);
}

// Widen half h of int8 row `row` of a [rows][128 B] tile written by TMA
// (128B swizzle: chunk c at c ^ (row & 7)), i.e. K values 64h .. 64h + 63,
// into row `row` of fp16 atom h of [2][rows][128 B], same swizzle (16-byte
// chunk j of an atom row at j ^ (row & 7)).
__device__ __forceinline__ void widen_half_row(uint32_t src, uint32_t dst, int rows, int row, int h) {
  const uint32_t sw = static_cast<uint32_t>(row & 7);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * h + cc;
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                 : "r"(src + static_cast<uint32_t>(row) * 128 + ((static_cast<uint32_t>(c) ^ sw) << 4)));
    uint32_t h[8];
    widen4(w0, h[0], h[1]);
    widen4(w1, h[2], h[3]);
    widen4(w2, h[4], h[5]);
    widen4(w3, h[6], h[7]);
    // K values 16c .. 16c + 15: atom c >> 2, fp16 chunks 2 (c & 3) and 2 (c & 3) + 1
    const uint32_t atom = dst + static_cast<uint32_t>((c >> 2) * rows * 128) + static_cast<uint32_t>(row) * 128;
    const uint32_t j0 = static_cast<uint32_t>(2 * (c & 3));
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(atom + ((j0 ^ sw) << 4)), "r"(h[0]), "r"(h[1]),
                 "r"(h[2]), "r"(h[3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(atom + (((j0 + 1) ^ sw) << 4)), "r"(h[4]), "r"(h[5]),
                 "r"(h[6]), "r"(h[7])
                 : "memory");
  }
}

template <int NA, bool RAW>
__global__ void __launch_bounds__(THREADS_T, 1) gemm_small_tc_kernel(const __grid_constant__ SmallTcParams p) {
  using C = SCfg<NA>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t base16 = sbase + static_cast<uint32_t>(p.stages * C::STAGE8);
  uint64_t* load_full = reinterpret_cast<uint64_t*>(smem + p.stages * C::STAGE8 + p.stages16 * C::STAGE16);
  uint64_t* src_free = load_full + MAX_STAGES8;  // converters have read the int8 tiles
  uint64_t* cvt_full = src_free + MAX_STAGES8;   // fp16 tiles written
  uint64_t* mma_done = cvt_full + MAX_STAGES16;  // MMAs of the stage complete: fp16 tiles free
  uint64_t* final_bar = mma_done + MAX_STAGES16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  int li = 0;
  while (li + 1 < p.outs.count && tile >= p.outs.o[li + 1].tile_begin) ++li;
  const GemmOut& out = p.outs.o[li];
  const int o0 = (tile - out.tile_begin) * WROWS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&load_full[s], 1);
      mbar_init(&src_free[s], CONV_WARPS);
    }
    for (int s = 0; s < p.stages16; ++s) {
      mbar_init(&cvt_full[s], CONV_WARPS);
      mbar_init(&mma_done[s], 1);
    }
    mbar_init(final_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the codes and scales come from the previous kernel of the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");

  auto stage_w8 = [&](int s) { return sbase + static_cast<uint32_t>(s * C::STAGE8); };
  auto stage_x8 = [&](int s) { return stage_w8(s) + C::W8; };
  auto stage_w16 = [&](int s) { return base16 + static_cast<uint32_t>(s * C::STAGE16); };
  auto stage_x16 = [&](int s) { return stage_w16(s) + C::W16; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int kt = 0; kt < p.ktiles; ++kt) {
        const int s = kt % p.stages, round = kt / p.stages;
        if (round > 0 && !mbar_wait_bounded(&src_free[s], (round - 1) & 1, p.spin_limit)) {
          record_status(CONVROT_ERR_TIMEOUT);
          break;
        }
        mbar_expect_tx(&load_full[s], WROWS * KT + NA * KT);
        tma_load_2d(stage_w8(s), &p.tmap_w[li], kt * KT, o0, &load_full[s]);
        tma_load_2d(stage_x8(s), &p.tmap_x, kt * KT, 0, &load_full[s]);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      bool ok = true;
      for (int kt = 0; kt < p.ktiles && ok; ++kt) {
        const int s = kt % p.stages16, round = kt / p.stages16;
        if (!mbar_wait_bounded(&cvt_full[s], round & 1, p.spin_limit)) {
          record_status(CONVROT_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const int chunk = kt / KCHUNK_TILES;
        const uint32_t d = tmem_base + static_cast<uint32_t>(chunk * NA);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t sa = stage_w16(s) + static_cast<uint32_t>(a * WROWS * 128 + k * 32);
            const uint32_t sb = stage_x16(s) + static_cast<uint32_t>(a * NA * 128 + k * 32);
            const uint32_t acc = (kt % KCHUNK_TILES != 0 || a > 0 || k > 0) ? 1u : 0u;
            tc_mma_f16(d, sw128_desc(sa), sw128_desc(sb), C::IDESC, acc);
          }
        tc_commit(&mma_done[s]);
      }
      tc_commit(final_bar);
    }
  } else {
    // ------------------------------------------- converters, then epilogue
    const int q = warp & 3;                  // TMEM lane quadrant this warp may read
    const int col_half = (warp - 2) >> 2;    // which half of the NA columns it reads
    const int wrow = q * 32 + lane;          // weight row of the tile this thread widens
    const int ct = threadIdx.x - 64;         // 0 .. 32 * CONV_WARPS - 1
    bool ok = true;
    for (int kt = 0; kt < p.ktiles; ++kt) {
      const int s8 = kt % p.stages, round8 = kt / p.stages;
      const int s16 = kt % p.stages16, round16 = kt / p.stages16;
      bool got = ok && mbar_wait_bounded(&load_full[s8], round8 & 1, p.spin_limit);
      if (got && round16 > 0) got = mbar_wait_bounded(&mma_done[s16], (round16 - 1) & 1, p.spin_limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0 && ok) record_status(CONVROT_ERR_TIMEOUT);
        ok = false;
        break;
      }
      widen_half_row(stage_w8(s8), stage_w16(s16), WROWS, wrow, col_half);
      for (int r = ct; r < 2 * NA; r += 32 * CONV_WARPS) widen_half_row(stage_x8(s8), stage_x16(s16), NA, r >> 1, r & 1);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> MMA reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&src_free[s8]);
        mbar_arrive(&cvt_full[s16]);
      }
    }
    // ---- epilogue: chunk sums in int32, then scale, bias, bf16
    const bool done = ok && mbar_wait_bounded(final_bar, 0, p.spin_limit);
    if (__all_sync(0xffffffffu, done)) {
      tc_fence_after();
      constexpr int HC = NA / 2;  // activation rows (TMEM columns) this warp reads
      int acc[HC];
#pragma unroll
      for (int j = 0; j < HC; ++j) acc[j] = 0;
      const int nch = (p.ktiles + KCHUNK_TILES - 1) / KCHUNK_TILES;
      for (int c = 0; c < nch; ++c) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(c * NA + col_half * HC);
#pragma unroll
        for (int j0 = 0; j0 < HC; j0 += 8) {
          uint32_t r[8];
          tc_ld_32x32b_x8(taddr + j0, r);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[j0 + e] += __float2int_rz(__uint_as_float(r[e]));
        }
      }
      const int o = o0 + wrow;
      if (o < out.n) {
        const float swo = RAW ? 0.0f : out.sw[o];
        const float bo = (!RAW && out.bias) ? out.bias[o] : 0.0f;
#pragma unroll
        for (int j = 0; j < HC; ++j) {
          const int r = col_half * HC + j;
          if (r < p.M) {
            if constexpr (RAW) {
              static_cast<int*>(out.y)[r * out.ldy + o] = acc[j];
            } else {
              static_cast<__nv_bfloat16*>(out.y)[r * out.ldy + o] =
                  __float2bfloat16_rn(fmaf(static_cast<float>(acc[j]), p.sx[r] * swo, bo));
            }
          }
        }
      }
    } else if (lane == 0) {
      record_status(CONVROT_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(p.tmem_cols)
                 : "memory");
  }
}

bool make_map_i8(EncodeTiledFn enc, CUtensorMap* map, const void* base, long long rows, int K, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(KT), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t tmem_columns(int cols) {
  uint32_t c = 32;
  while (static_cast<int>(c) < cols) c <<= 1;
  return c;
}

template <int NA, bool RAW>
cudaError_t launch_small_tc(EncodeTiledFn enc, const int8_t* Qx, const float* sx, long long M, int K,
                            GemmOutputs outs, cudaStream_t st) {
  using C = SCfg<NA>;
  SmallTcParams p;
  memset(&p, 0, sizeof(p));
  if (!make_map_i8(enc, &p.tmap_x, Qx, M, K, NA)) return cudaErrorInvalidValue;
  int nt = 0;
  for (int i = 0; i < outs.count; ++i) {
    outs.o[i].tile_begin = nt;
    nt += (outs.o[i].n + WROWS - 1) / WROWS;
    if (!make_map_i8(enc, &p.tmap_w[i], outs.o[i].qw, outs.o[i].n, K, WROWS)) return cudaErrorInvalidValue;
  }
  p.outs = outs;
  p.sx = sx;
  p.M = M;
  p.K = K;
  p.ktiles = K / KT;
  const int nch = (p.ktiles + KCHUNK_TILES - 1) / KCHUNK_TILES;
  p.tmem_cols = tmem_columns(nch * NA);
  const int bar_bytes = (2 * MAX_STAGES8 + 2 * MAX_STAGES16 + 1) * 8 + 8;
  const int budget = 232448 - 1024 - bar_bytes;
  // the deepest fp16 ring that still leaves three int8 stages (or all of K)
  p.stages16 = std::min(p.ktiles, MAX_STAGES16);
  while (p.stages16 > 2 && budget - p.stages16 * C::STAGE16 < std::min(3, p.ktiles) * C::STAGE8) --p.stages16;
  p.stages = std::min(p.ktiles, std::min(MAX_STAGES8, (budget - p.stages16 * C::STAGE16) / C::STAGE8));
  if (p.stages < 1) return cudaErrorInvalidConfiguration;
  p.spin_limit = kDefaultSpinLimit;
  const int smem = 1024 + p.stages * C::STAGE8 + p.stages16 * C::STAGE16 + bar_bytes;
  auto kern = gemm_small_tc_kernel<NA, RAW>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nt);
  cfg.blockDim = dim3(THREADS_T);
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

int status_word_gemm_small_tc() { return status_word_small_tc_local(); }

// 17..64 rows (measured on GB300: up to 16 rows the int8 mma.sync stream of
// gemm_small is faster, beyond it this kernel is 1.5-3x faster), K a multiple
// of 128, and every exact chunk of NA columns fits the 512 columns of tensor
// memory.
bool gemm_small_tc_supported(long long M, int K) {
  if (M <= 16 || M > 64 || K % KT != 0 || K < KT) return false;
  const int na = static_cast<int>((M + 15) / 16) * 16;
  const int nch = (K / KT + KCHUNK_TILES - 1) / KCHUNK_TILES;
  return nch * na <= 512;
}

cudaError_t gemm_small_tc_launch(const int8_t* Qx, const float* sx, long long M, int K, const GemmOutputs& outs,
                                 bool raw, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  if (M <= 16) return raw ? launch_small_tc<16, true>(enc, Qx, sx, M, K, outs, st)
                          : launch_small_tc<16, false>(enc, Qx, sx, M, K, outs, st);
  if (M <= 32) return raw ? launch_small_tc<32, true>(enc, Qx, sx, M, K, outs, st)
                          : launch_small_tc<32, false>(enc, Qx, sx, M, K, outs, st);
  if (M <= 48) return raw ? launch_small_tc<48, true>(enc, Qx, sx, M, K, outs, st)
                          : launch_small_tc<48, false>(enc, Qx, sx, M, K, outs, st);
  return raw ? launch_small_tc<64, true>(enc, Qx, sx, M, K, outs, st)
             : launch_small_tc<64, false>(enc, Qx, sx, M, K, outs, st);
}

}  // namespace convrot
