// Rotate + row-absmax + quantize with the rotation applied as a dense matmul
// on the tensor cores ("feat: load ConvRot int4 and per-channel int8
// safetensors", section "The rotation": the rotation applied as one matmul
// against a shared constant). It computes what the butterfly kernels compute
// and exists to compare the two on the same hardware.
//
// X (bf16, dense [M, K]) is viewed as segments of S = max(G, 64) elements:
// A = X as [M*K/S, S]. The constant B (S x S, bf16) is the sign pattern of the
// unnormalized rotation, I_{S/G} (x) (2^n R_G), entries +-1 and 0, exact in
// bf16; D = A B^T lands in tensor memory in fp32 (tcgen05.mma kind::f16,
// M = 128, N = S). Like the butterfly kernels it drops the 2^-n factor and
// folds it into the stored scale. A tile is 128 segments holding whole rows,
// so the row absmax never leaves the CTA.
//
// Roles (persistent, 160 threads): warps 0-3 are the epilogue (TMEM lane
// quadrants 0-3): absmax, a 128-thread named barrier, then quantize and
// store straight from TMEM. Warp 4 allocates TMEM, issues the A-tile TMA and
// the MMAs. The A buffer is refilled as soon as the MMAs of the previous tile
// have read it, and two TMEM accumulators alternate, so loads overlap the
// epilogue. Every wait is bounded and reports CONVROT_ERR_TIMEOUT.
#include <algorithm>

#include "common.cuh"
#include "tc_common.cuh"

namespace convrot {

namespace {

using namespace tc;

CONVROT_DEFINE_STATUS_WORD(status_word_hmatmul_local)

constexpr int HM_THREADS = 160;

template <int G>
struct HmCfg {
  static constexpr int S = G < 64 ? 64 : G;         // segment = MMA N = reduction length
  static constexpr int KB = S / 64;                 // 64-element k-blocks
  static constexpr int A_BYTES = KB * 128 * 128;    // 128 rows x 128 B per k-block
  static constexpr int B_BYTES = KB * S * 128;      // S rows x 128 B per k-block
  static constexpr int TMEM_COLS = 2 * S < 32 ? 32 : 2 * S;
  static constexpr uint32_t IDESC = idesc_f16(128, S, true);
  static constexpr int N = ilog4_c(G);
};

// +1 / -1 / 0 entry (n, k) of I_{S/G} (x) (2^n R_G): -1 for every base-4
// digit position where the digits of n and k add up to 3.
template <int G>
__device__ __forceinline__ float sign_entry(int n, int k) {
  if ((n / G) != (k / G)) return 0.0f;
  int neg = 0;
#pragma unroll
  for (int d = 0; d < HmCfg<G>::N; ++d) neg ^= (((n >> (2 * d)) & 3) + ((k >> (2 * d)) & 3)) == 3;
  return neg ? -1.0f : 1.0f;
}

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

template <int G>
__global__ void __launch_bounds__(HM_THREADS, 1)
    hmatmul_kernel(const __grid_constant__ CUtensorMap amap, long long M, int K, int rows_per_tile, int arows,
                   int8_t* __restrict__ Q, float* __restrict__ S, __half* __restrict__ Q16, float s_div,
                   long long spin_limit) {
  using C = HmCfg<G>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t a_base = smem_u32(smem);
  const uint32_t b_base = a_base + C::A_BYTES;
  unsigned int* rowmax_buf = reinterpret_cast<unsigned int*>(smem + C::A_BYTES + C::B_BYTES);  // [3][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(rowmax_buf + 3 * 128);
  uint64_t* a_full = bars + 0;
  uint64_t* a_empty = bars + 1;
  uint64_t* acc_full = bars + 2;   // [2]
  uint64_t* acc_empty = bars + 4;  // [2]
  uint64_t* final_bar = bars + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int segs_per_row = K / C::S;
  const long long ntiles = (M + rows_per_tile - 1) / rows_per_tile;

  // the constant operand, in the 128B-swizzled K-major layout the MMA reads
  for (int idx = threadIdx.x; idx < C::S * C::S / 8; idx += HM_THREADS) {
    const int n = idx / (C::S / 8);
    const int kc = idx % (C::S / 8);  // 8-element chunk along k
    const int kb = kc >> 3, c = kc & 7;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 p =
          __floats2bfloat162_rn(sign_entry<G>(n, kc * 8 + 2 * e), sign_entry<G>(n, kc * 8 + 2 * e + 1));
      w[e] = *reinterpret_cast<const uint32_t*>(&p);
    }
    const uint32_t off = static_cast<uint32_t>(kb * C::S * 128 + n * 128 + ((c ^ (n & 7)) << 4));
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(b_base + off), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
  }
  for (int i = threadIdx.x; i < 3 * 128; i += HM_THREADS) rowmax_buf[i] = 0u;
  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // generic-proxy writes of B become visible to the tensor cores
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
        // A buffer free once the previous tile's MMAs have read it
        if (!mbar_wait_bounded(a_empty, (it & 1) ^ 1, spin_limit)) { ok = false; break; }
        // the box is `arows` rows of every k-block (rows beyond are never used)
        mbar_expect_tx(a_full, static_cast<uint32_t>(C::KB * arows * 128));
        const int row0 = static_cast<int>(t * rows_per_tile) * segs_per_row;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) tma_load_2d(a_base + kb * 128 * 128, &amap, kb * 64, row0, a_full);
        const int b = it & 1, u = it >> 1;
        if (!mbar_wait_bounded(&acc_empty[b], (u & 1) ^ 1, spin_limit)) { ok = false; break; }
        if (!mbar_wait_bounded(a_full, it & 1, spin_limit)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * C::S);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc_mma_f16(d, sw128_desc(a_base + kb * 128 * 128 + k * 32), sw128_desc(b_base + kb * C::S * 128 + k * 32),
                       C::IDESC, (kb > 0 || k > 0) ? 1u : 0u);
        tc_commit(a_empty);
        tc_commit(&acc_full[b]);
      }
      if (!ok) {
        record_status(CONVROT_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit(final_bar);
      if (!mbar_wait_bounded(final_bar, 0, spin_limit)) record_status(CONVROT_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int sidx = warp * 32 + lane;  // segment (TMEM lane) within the tile
    const int rr = sidx / segs_per_row;
    const int col0 = (sidx % segs_per_row) * C::S;
    const bool valid_seg = sidx < arows;
    int it = 0;
    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
      const int b = it & 1, u = it >> 1;
      unsigned int* rowmax = rowmax_buf + (it % 3) * 128;
      // After a failed wait anywhere in the CTA the epilogue stops waiting but
      // keeps iterating (on stale data, with the error recorded), so that all
      // four warps keep meeting at the named barrier below.
      const bool got = !*abort_flag && mbar_wait_bounded(&acc_full[b], u & 1, spin_limit);
      if (!__all_sync(0xffffffffu, got) && lane == 0) {
        record_status(CONVROT_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(b * C::S);
      float m = 0.0f;
#pragma unroll
      for (int c = 0; c < C::S / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + c * 32, r);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) m = fmax3(m, fabsf(__uint_as_float(r[e])), fabsf(__uint_as_float(r[e + 1])));
      }
      if (valid_seg) atomicMax(&rowmax[rr], __float_as_uint(m));
      named_bar(1, 128);
      // buffer (it + 2) % 3 was last read two tiles ago, before this barrier
      if (threadIdx.x < 128) rowmax_buf[((it + 2) % 3) * 128 + threadIdx.x] = 0u;
      const long long row = t * rows_per_tile + rr;
      const bool store = valid_seg && row < M;
      const float amax = valid_seg ? __uint_as_float(rowmax[rr]) : 0.0f;
      const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
      const float2 inv2 = make_float2(inv, inv);
      const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
#pragma unroll
      for (int c = 0; c < C::S / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + c * 32, r);
        tc_wait_ld();
        uint32_t words[8], hw[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 t01 = f2_fma(make_float2(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1])), inv2, mg2);
          const float2 t23 =
              f2_fma(make_float2(__uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])), inv2, mg2);
          const uint32_t b01 = __byte_perm(__float_as_uint(t01.x), __float_as_uint(t01.y), 0x0040);
          const uint32_t b23 = __byte_perm(__float_as_uint(t23.x), __float_as_uint(t23.y), 0x0040);
          words[k] = __byte_perm(b01, b23, 0x5410);
          const float2 c01 = f2_sub(t01, mg2), c23 = f2_sub(t23, mg2);
          const __half2 h01 = __floats2half2_rn(c01.x, c01.y);
          const __half2 h23 = __floats2half2_rn(c23.x, c23.y);
          hw[2 * k] = *reinterpret_cast<const uint32_t*>(&h01);
          hw[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&h23);
        }
        if (store) {
          const long long e = row * static_cast<long long>(K) + col0 + 32 * c;
          stg_256(Q + e, words);
          if (Q16) {
            const uint32_t(&h0)[8] = *reinterpret_cast<const uint32_t(*)[8]>(hw);
            const uint32_t(&h1)[8] = *reinterpret_cast<const uint32_t(*)[8]>(hw + 8);
            stg_256(Q16 + e, h0);
            stg_256(Q16 + e + 16, h1);
          }
        }
      }
      if (store && col0 == 0) S[row] = amax / s_div;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS) : "memory");
  }
}

template <int G>
cudaError_t launch_hm(const void* X, long long M, int K, int8_t* Q, float* S, uint16_t* Q16, cudaStream_t st) {
  using C = HmCfg<G>;
  const int segs_per_row = K / C::S;
  if (K % C::S != 0 || segs_per_row > 128) return cudaErrorInvalidValue;
  const int rows_per_tile = 128 / segs_per_row;
  const int arows = rows_per_tile * segs_per_row;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  // A = X as [M*K/S, S] bf16; one box = 64 columns of `arows` segments
  CUtensorMap map;
  const long long nseg = M * segs_per_row;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(C::S), static_cast<cuuint64_t>(nseg)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(C::S) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(arows)};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int smem = 1024 + C::A_BYTES + C::B_BYTES + 3 * 128 * 4 + 8 * 8 + 16;
  auto kern = hmatmul_kernel<G>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(reinterpret_cast<const void*>(kern), HM_THREADS, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // tensor memory: at most 512 columns per SM in total
  per_sm = std::min(per_sm, 512 / C::TMEM_COLS);
  const long long ntiles = (M + rows_per_tile - 1) / rows_per_tile;
  const long long grid = std::min<long long>(ntiles, static_cast<long long>(per_sm) * device_sm_count());
  kern<<<static_cast<unsigned>(grid), HM_THREADS, smem, st>>>(map, M, K, rows_per_tile, arows, Q, S,
                                                               reinterpret_cast<__half*>(Q16),
                                                               127.0f * static_cast<float>(1 << C::N), kDefaultSpinLimit);
  return cudaGetLastError();
}

}  // namespace

int status_word_hmatmul() { return status_word_hmatmul_local(); }

bool hmatmul_supported(long long K, long long ldx, int G) {
  const int S = G < 64 ? 64 : G;
  return (G == 16 || G == 64 || G == 256) && ldx == K && K % S == 0 && K / S <= 128;
}

cudaError_t hmatmul_launch(const void* X, long long M, int K, long long ldx, int G, int8_t* Q, float* S,
                           uint16_t* Q16, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (!hmatmul_supported(K, ldx, G)) return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(Q) % 32 || reinterpret_cast<uintptr_t>(Q16) % 32) return cudaErrorMisalignedAddress;
  switch (G) {
    case 16: return launch_hm<16>(X, M, K, Q, S, Q16, st);
    case 64: return launch_hm<64>(X, M, K, Q, S, Q16, st);
    default: return launch_hm<256>(X, M, K, Q, S, Q16, st);
  }
}

}  // namespace convrot
