// Fused rotate + row-absmax + quantize kernels.
//
// Method ("INT8 Convrot Safetensors", sections "How INT8 convrot works" and
// "Runtime activation quantization"): every contiguous group of G input
// features of a row is multiplied by R_G, the normalized Kronecker power of
// H4 (G = 4^n); then s[r] = max|X_rot[r,:]| / 127 and
// Q = clamp(round(X_rot / s), -127, 127). The block randomized Hadamard
// variant (gemma.cpp issue "Add experimental W8A8 MatMul with optional
// QuaRot-style rotation", section "Rotation method") multiplies by +-1 signs,
// applies a Walsh-Hadamard transform and scales by 1/sqrt(B).
//
// Arithmetic shared by both kernels here (they give bit-identical results):
//  * The butterfly is unnormalized. One radix-4 stage maps (x0,x1,x2,x3) to
//    2*H4*x via u01=x0+x1, w0=x0-x1, u23=x2+x3, w2=x2-x3 and
//    (u01+w2, u01-w2, u23+w0, u23-w0); row a of 2*H4 is all +1 except -1 in
//    column 3-a. Digits are processed from the least significant one up.
//    The dropped factor c (2^-n, or 1/sqrt(B)) scales every element of the
//    row alike, so the codes do not depend on it; it is folded into the
//    stored scale: s = amax / (127 / c).
//  * inv = 127 / amax (IEEE division) and the code is round(y * inv) with
//    one rounding (see kRoundMagic). |y| <= amax, so |y * inv| < 127.5 and
//    the clamp to [-127, 127] can never bite; a zero row gets inv = 0,
//    codes 0 and scale 0.
#include <algorithm>
#include <cstdio>

#include "common.cuh"

namespace convrot {

CONVROT_DEFINE_STATUS_WORD(status_word_rotquant)

__device__ __forceinline__ void h4_stage(float& x0, float& x1, float& x2, float& x3) {
  const float u01 = x0 + x1, w0 = x0 - x1, u23 = x2 + x3, w2 = x2 - x3;
  x0 = u01 + w2;
  x1 = u01 - w2;
  x2 = u23 + w0;
  x3 = u23 - w0;
}

__device__ __forceinline__ void h4_stage(float2& x0, float2& x1, float2& x2, float2& x3) {
  const float2 u01 = f2_add(x0, x1), w0 = f2_sub(x0, x1), u23 = f2_add(x2, x3), w2 = f2_sub(x2, x3);
  x0 = f2_add(u01, w2);
  x1 = f2_sub(u01, w2);
  x2 = f2_add(u23, w0);
  x3 = f2_sub(u23, w0);
}

// ============================================================ generic ======
// One CTA per row (grid-stride); the row lives in shared memory as fp32 and
// every radix stage is one pass over it. Handles every transform, any
// supported G, fp32 or bf16 input and any alignment.

template <typename Tin>
__device__ __forceinline__ float load_in(const Tin* p);
template <>
__device__ __forceinline__ float load_in<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_in<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename Tin>
__global__ void __launch_bounds__(256) rq_generic_kernel(const Tin* __restrict__ X, long long M, int K, long long ldx,
                                                         int transform, int G, const int8_t* __restrict__ signs,
                                                         int8_t* __restrict__ Q, float* __restrict__ S,
                                                         __half* __restrict__ Q16, float s_div) {
  extern __shared__ float buf[];
  __shared__ float red[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  for (long long row = blockIdx.x; row < M; row += gridDim.x) {
    const Tin* x = X + row * ldx;
    for (int i = tid; i < K; i += nt) {
      float v = load_in(x + i);
      if (transform == CONVROT_T_RHT && signs[i & (G - 1)] < 0) v = -v;
      buf[i] = v;
    }
    __syncthreads();
    if (transform == CONVROT_T_REGULAR_H4) {
      for (int stride = 1; stride < G; stride *= 4) {
        for (int q = tid; q < K / 4; q += nt) {
          const int lo = q % stride, hi = q / stride;
          const int i0 = hi * 4 * stride + lo;
          float x0 = buf[i0], x1 = buf[i0 + stride], x2 = buf[i0 + 2 * stride], x3 = buf[i0 + 3 * stride];
          h4_stage(x0, x1, x2, x3);
          buf[i0] = x0;
          buf[i0 + stride] = x1;
          buf[i0 + 2 * stride] = x2;
          buf[i0 + 3 * stride] = x3;
        }
        __syncthreads();
      }
    } else if (transform == CONVROT_T_RHT) {
      for (int stride = 1; stride < G; stride *= 2) {
        for (int p = tid; p < K / 2; p += nt) {
          const int lo = p % stride, hi = p / stride;
          const int i0 = hi * 2 * stride + lo;
          const float a = buf[i0], b = buf[i0 + stride];
          buf[i0] = a + b;
          buf[i0 + stride] = a - b;
        }
        __syncthreads();
      }
    }
    float m = 0.0f;
    for (int i = tid; i < K; i += nt) m = fmaxf(m, fabsf(buf[i]));
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    if (tid < 32) {
      m = tid < (nt >> 5) ? red[tid] : 0.0f;
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (tid == 0) red[0] = m;
    }
    __syncthreads();
    const float amax = red[0];
    const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
    int8_t* q = Q + row * (long long)K;
    for (int i = tid; i < K; i += nt) {
      const int c = code_from_magic(fmaf(buf[i], inv, kRoundMagic));
      q[i] = static_cast<int8_t>(c);
      if (Q16) Q16[row * (long long)K + i] = __int2half_rn(c);
    }
    if (tid == 0) S[row] = amax / s_div;
    __syncthreads();
  }
}

// =============================================================== fast ======
// Fast kernel for bf16 input and the regular Hadamard.
//
// A CTA owns a tile of R consecutive rows (persistent grid-stride loop).
//  Phase R: each thread takes SEGS segments of G1 consecutive elements,
//    loaded with 32-byte loads (a warp reads 1 KB contiguous per load), and
//    runs the radix-4 stages of the low digits in registers (G1 = 16: two
//    digits, G1 = 64: three). The loads of the next tile are issued as soon
//    as these registers are free.
//  Phase C (G > G1): the rotated segments are parked in shared memory as
//    fp32 (XOR-swizzled against bank conflicts), where the row stays across
//    the reduction. Each thread then runs the high digits on units of
//    G2 = G/G1 rows x 2 adjacent columns of the group seen as a G2 x G1
//    matrix, two columns per packed fp32x2 operation, and writes the unit
//    back in place.
//  Row absmax: a warp reduction over the lanes of each row (lanes of one
//    warp may straddle two rows), then one shared-memory atomicMax.
//  Quantize: in the load layout again, so the int8 codes (16-byte stores)
//    and the fp16 copies (32-byte stores) leave coalesced, straight to HBM.
// With G <= 16 a segment holds whole groups and nothing leaves registers.

template <int G, int G1, int SEGS>
struct FastCfg {
  static constexpr int G2 = G > G1 ? G / G1 : 1;
  static constexpr int ND1 = ilog4_c(G < G1 ? G : G1);
  static constexpr int ND2 = ilog4_c(G2);
  static constexpr int EPT = SEGS * G1;
  static constexpr bool PHASE_C = G2 > 1;
  static constexpr int NU = PHASE_C ? EPT / (2 * G2) : 0;  // phase-C units per thread
  static constexpr int LOADS = G1 / 16;
};

// fp32 buffer: 16-byte chunk index -> physical chunk (a bijection inside each
// aligned block of 8 chunks).
template <int G, int G1>
__device__ __forceinline__ int swz_chunk(int c) {
  if constexpr (G1 == 16) {
    constexpr int GS = ilog2_c(G / 4 > 1 ? G / 4 : 2);
    return c ^ ((c >> 3) & 7) ^ (((c >> GS) & 1) << 2);
  } else {
    return c ^ ((c >> 4) & 7);
  }
}
// Quantize N consecutive values of one row (N a multiple of 16) and store the
// codes (16-byte stores) and, if requested, their fp16 copies (32-byte
// stores) at dense element offset e, if e lies inside the matrix.
template <int N>
__device__ __forceinline__ void quantize_store(const float (&p)[N], float inv, long long e, long long total_elems,
                                               int8_t* __restrict__ Q, __half* __restrict__ Q16) {
  const float2 inv2 = make_float2(inv, inv);
  const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
#pragma unroll
  for (int k16 = 0; k16 < N / 16; ++k16) {
    uint32_t words[4];
    uint32_t hw[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int o = 16 * k16 + 4 * k;
      const float2 t01 = f2_fma(make_float2(p[o], p[o + 1]), inv2, mg2);
      const float2 t23 = f2_fma(make_float2(p[o + 2], p[o + 3]), inv2, mg2);
      const uint32_t b01 = __byte_perm(__float_as_uint(t01.x), __float_as_uint(t01.y), 0x0040);
      const uint32_t b23 = __byte_perm(__float_as_uint(t23.x), __float_as_uint(t23.y), 0x0040);
      words[k] = __byte_perm(b01, b23, 0x5410);
      if (Q16) {
        const float2 c01 = f2_sub(t01, mg2), c23 = f2_sub(t23, mg2);
        const __half2 h01 = __floats2half2_rn(c01.x, c01.y);
        const __half2 h23 = __floats2half2_rn(c23.x, c23.y);
        hw[2 * k] = *reinterpret_cast<const uint32_t*>(&h01);
        hw[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&h23);
      }
    }
    if (e < total_elems) {
      stg_128(Q + e + 16 * k16, make_uint4(words[0], words[1], words[2], words[3]));
      if (Q16) stg_256(Q16 + e + 16 * k16, hw);
    }
  }
}

template <int G, int G1, int SEGS>
__global__ void __launch_bounds__(384) rq_fast_kernel(const __nv_bfloat16* __restrict__ X, long long M, int K,
                                                       long long ldx, int R, int NT, int8_t* __restrict__ Q,
                                                       float* __restrict__ S, __half* __restrict__ Q16,
                                                       float s_div, int fbytes) {
  using C = FastCfg<G, G1, SEGS>;
  extern __shared__ __align__(128) unsigned char smem[];
  float* fbuf = reinterpret_cast<float*>(smem);
  unsigned int* rowmax_buf = reinterpret_cast<unsigned int*>(smem + fbytes);  // [2][R]

  const int tid = threadIdx.x, lane = tid & 31;
  const bool active = tid < NT;
  const long long ntiles = (M + R - 1) / R;
  const int tile_elems = R * K;
  const long long total_elems = M * static_cast<long long>(K);

  // Tile-invariant geometry, computed once: the row of each of this
  // thread's segments and its offset in X. The outputs are dense [M, K], so
  // their offsets need no row / column split.
  int seg_row[SEGS];
  long long seg_xoff[SEGS];
#pragma unroll
  for (int j = 0; j < SEGS; ++j) {
    const int e = (tid + j * NT) * G1;
    seg_row[j] = e / K;
    seg_xoff[j] = seg_row[j] * ldx + (e - seg_row[j] * K);
  }
  // Phase-C units: G2 rows x 2 adjacent columns of one group matrix.
  int unit_base[C::NU > 0 ? C::NU : 1];
  int unit_row[C::NU > 0 ? C::NU : 1];
  if constexpr (C::PHASE_C) {
    const int groups = K / G;
#pragma unroll
    for (int i = 0; i < C::NU; ++i) {
      const int b = tid + i * NT;
      const int cp = b % (G1 / 2);
      const int rest = b / (G1 / 2);
      const int g = rest % groups;
      const int r = rest / groups;
      unit_row[i] = r;
      unit_base[i] = r * K + g * G + 2 * cp;
    }
  }

  U32x8 raw[SEGS][C::LOADS];
  auto issue_loads = [&](long long tile) {
    const long long rbase = tile * R;
    const __nv_bfloat16* xt = X + rbase * ldx;
#pragma unroll
    for (int j = 0; j < SEGS; ++j) {
      const bool ok = active && rbase + seg_row[j] < M;
#pragma unroll
      for (int l = 0; l < C::LOADS; ++l) {
        if (ok) {
          raw[j][l] = ldg_nc_256(xt + seg_xoff[j] + 16 * l);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) raw[j][l].w[k] = 0u;
        }
      }
    }
  };

  // Row maxima are double-buffered by iteration parity: the buffer of the
  // next iteration is cleared during this one, after every read of it by the
  // previous iteration has passed that iteration's final barrier.
  for (int i = tid; i < 2 * R; i += blockDim.x) rowmax_buf[i] = 0u;
  __syncthreads();

  long long tile = blockIdx.x;
  if (tile < ntiles) issue_loads(tile);

  for (int it = 0; tile < ntiles; tile += gridDim.x, ++it) {
    unsigned int* rowmax = rowmax_buf + (it & 1) * R;
    for (int i = tid; i < R; i += blockDim.x) rowmax_buf[((it + 1) & 1) * R + i] = 0u;
    const long long tile_off = tile * static_cast<long long>(tile_elems);
    const long long next = tile + gridDim.x;

    if constexpr (C::PHASE_C) {
      // ---- phase R: widen, low-digit stages, park the row in shared memory
      if (active) {
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
          float v[G1];
#pragma unroll
          for (int l = 0; l < C::LOADS; ++l)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[l * 16 + 2 * k] = bf16lo_f32(raw[j][l].w[k]);
              v[l * 16 + 2 * k + 1] = bf16hi_f32(raw[j][l].w[k]);
            }
#pragma unroll
          for (int d = 0; d < C::ND1; ++d) {
            const int st = 1 << (2 * d);
#pragma unroll
            for (int base = 0; base < G1; base += 4 * st)
#pragma unroll
              for (int o = 0; o < st; ++o) h4_stage(v[base + o], v[base + o + st], v[base + o + 2 * st], v[base + o + 3 * st]);
          }
          const int c0 = ((tid + j * NT) * G1) >> 2;
#pragma unroll
          for (int k = 0; k < G1 / 4; ++k)
            reinterpret_cast<float4*>(fbuf)[swz_chunk<G, G1>(c0 + k)] =
                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
      }
      // the raw registers are free: start the next tile's loads now
      if (next < ntiles) issue_loads(next);
      __syncthreads();

      // ---- phase C: high-digit stages in place, two columns per packed op
      float m_unit[C::NU];
#pragma unroll
      for (int i = 0; i < C::NU; ++i) {
        float m = 0.0f;
        if (active) {
          float2 w[C::G2];
          int addr[C::G2];
#pragma unroll
          for (int h = 0; h < C::G2; ++h) {
            const int e = unit_base[i] + h * G1;
            addr[h] = 2 * swz_chunk<G, G1>(e >> 2) + ((e >> 1) & 1);  // float2 slot
            w[h] = reinterpret_cast<const float2*>(fbuf)[addr[h]];
          }
#pragma unroll
          for (int d = 0; d < C::ND2; ++d) {
            const int st = 1 << (2 * d);
#pragma unroll
            for (int base = 0; base < C::G2; base += 4 * st)
#pragma unroll
              for (int o = 0; o < st; ++o)
                h4_stage(w[base + o], w[base + o + st], w[base + o + 2 * st], w[base + o + 3 * st]);
          }
#pragma unroll
          for (int h = 0; h < C::G2; ++h) {
            reinterpret_cast<float2*>(fbuf)[addr[h]] = w[h];
            m = fmax3(m, fabsf(w[h].x), fabsf(w[h].y));
          }
        }
        m_unit[i] = m;
      }
      // per-row absmax: warp max over lanes of the same row, one atomic each
#pragma unroll
      for (int i = 0; i < C::NU; ++i) {
        const int row = active ? unit_row[i] : -1;
        const unsigned grp = __match_any_sync(0xffffffffu, row);
        const unsigned mx = __reduce_max_sync(grp, __float_as_uint(m_unit[i]));
        if (active && lane == __ffs(grp) - 1) atomicMax(&rowmax[row], mx);
      }
      __syncthreads();

      // ---- quantize in the load layout: coalesced stores straight to HBM
      if (active) {
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
          const int seg = tid + j * NT;
          const float amax = __uint_as_float(rowmax[seg_row[j]]);
          const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
          const int c0 = (seg * G1) >> 2;
#pragma unroll
          for (int s16 = 0; s16 < G1 / 16; ++s16) {
            float v[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float4 f = reinterpret_cast<const float4*>(fbuf)[swz_chunk<G, G1>(c0 + 4 * s16 + k)];
              v[4 * k] = f.x;
              v[4 * k + 1] = f.y;
              v[4 * k + 2] = f.z;
              v[4 * k + 3] = f.w;
            }
            quantize_store<16>(v, inv, tile_off + static_cast<long long>(seg) * G1 + 16 * s16, total_elems, Q, Q16);
          }
        }
      }
    } else {
      // ---- G <= 16: a segment holds whole groups; everything stays in registers
      float v[SEGS][G1];
#pragma unroll
      for (int j = 0; j < SEGS; ++j)
#pragma unroll
        for (int l = 0; l < C::LOADS; ++l)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[j][l * 16 + 2 * k] = bf16lo_f32(raw[j][l].w[k]);
            v[j][l * 16 + 2 * k + 1] = bf16hi_f32(raw[j][l].w[k]);
          }
      if (next < ntiles) issue_loads(next);
#pragma unroll
      for (int d = 0; d < C::ND1; ++d) {
        const int st = 1 << (2 * d);
#pragma unroll
        for (int j = 0; j < SEGS; ++j)
#pragma unroll
          for (int base = 0; base < G1; base += 4 * st)
#pragma unroll
            for (int o = 0; o < st; ++o)
              h4_stage(v[j][base + o], v[j][base + o + st], v[j][base + o + 2 * st], v[j][base + o + 3 * st]);
      }
#pragma unroll
      for (int j = 0; j < SEGS; ++j) {
        float m = 0.0f;
        if (active) {
#pragma unroll
          for (int e = 0; e < G1; e += 2) m = fmax3(m, fabsf(v[j][e]), fabsf(v[j][e + 1]));
        }
        const int row = active ? seg_row[j] : -1;
        const unsigned grp = __match_any_sync(0xffffffffu, row);
        const unsigned mx = __reduce_max_sync(grp, __float_as_uint(m));
        if (active && lane == __ffs(grp) - 1) atomicMax(&rowmax[row], mx);
      }
      __syncthreads();
      if (active) {
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
          const float amax = __uint_as_float(rowmax[seg_row[j]]);
          const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
          quantize_store<G1>(v[j], inv, tile_off + static_cast<long long>(tid + j * NT) * G1, total_elems, Q, Q16);
        }
      }
    }
    for (int i = tid; i < R; i += blockDim.x)
      if (tile * R + i < M) S[tile * R + i] = __uint_as_float(rowmax[i]) / s_div;
    __syncthreads();
  }
}

// ================================================================ host =====

static float scale_divisor(int transform, int G) {
  if (transform == CONVROT_T_REGULAR_H4) return 127.0f * static_cast<float>(1 << (ilog2_c(G) / 2));
  if (transform == CONVROT_T_RHT) return static_cast<float>(127.0 * std::sqrt(static_cast<double>(G)));
  return 127.0f;
}


// Rows per tile: the smallest R for which R*K/EPT threads fill whole warps
// (or nearly), within the thread and shared-memory limits.
static bool choose_rows(int K, int ept, bool phase_c, int* R_out, int* NT_out) {
  int bestR = -1, bestNT = 0;
  double best_eff = -1.0;
  for (int R = 1; R <= 64; ++R) {
    if ((static_cast<long long>(R) * K) % ept) continue;
    const int NT = static_cast<int>(static_cast<long long>(R) * K / ept);
    if (NT > 384) break;
    if (phase_c && static_cast<long long>(R) * K * 4 > 96 * 1024) break;
    const int pad = (NT + 31) / 32 * 32;
    const double eff = static_cast<double>(NT) / pad;
    if (NT >= 96 && eff >= 0.95) {
      *R_out = R;
      *NT_out = NT;
      return true;
    }
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      bestR = R;
      bestNT = NT;
    }
  }
  if (bestR < 0) return false;
  *R_out = bestR;
  *NT_out = bestNT;
  return true;
}

template <int G, int G1, int SEGS>
static cudaError_t launch_fast(const __nv_bfloat16* X, long long M, int K, long long ldx, int8_t* Q, float* S,
                               __half* Q16, cudaStream_t st, bool* launched) {
  using C = FastCfg<G, G1, SEGS>;
  *launched = false;
  int R = 0, NT = 0;
  if (!choose_rows(K, C::EPT, C::PHASE_C, &R, &NT)) return cudaSuccess;
  const int threads = (NT + 31) / 32 * 32;
  // fp32 tile buffer (rounded up to whole swizzle blocks), then the row maxima
  const int fbytes = C::PHASE_C ? ((R * K * 4 + 511) / 512) * 512 : 0;
  const int smem = fbytes + 2 * R * 4;
  auto kern = rq_fast_kernel<G, G1, SEGS>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(reinterpret_cast<const void*>(kern), threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaSuccess;
  const long long tiles = (M + R - 1) / R;
  const long long grid = std::min<long long>(tiles, static_cast<long long>(per_sm) * device_sm_count());
  kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(X, M, K, ldx, R, NT, Q, S, Q16,
                                                             scale_divisor(CONVROT_T_REGULAR_H4, G), fbytes);
  *launched = true;
  return cudaGetLastError();
}

// Entry used by the ABI layer. Returns a cudaError_t; *path tells which
// kernel ran (0 = generic, 1 = fast).
cudaError_t rotquant_launch(const void* X, int in_dtype, long long M, int K, long long ldx, int G, int transform,
                            const int8_t* signs, int8_t* Q, float* S, uint16_t* Q16, int force_generic,
                            cudaStream_t st, int* path) {
  *path = 0;
  if (M <= 0) return cudaSuccess;
  __half* q16 = reinterpret_cast<__half*>(Q16);
  const bool aligned32 = (reinterpret_cast<uintptr_t>(X) % 32 == 0) && (ldx % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(Q) % 16 == 0) &&
                         (Q16 == nullptr || reinterpret_cast<uintptr_t>(Q16) % 16 == 0);
  if (!force_generic && in_dtype == CONVROT_DTYPE_BF16 && transform == CONVROT_T_REGULAR_H4 && aligned32 &&
      K % 16 == 0) {
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(X);
    bool launched = false;
    cudaError_t e = cudaSuccess;
    switch (G) {
      case 4: e = launch_fast<4, 16, 2>(xb, M, K, ldx, Q, S, q16, st, &launched); break;
      case 16: e = launch_fast<16, 16, 2>(xb, M, K, ldx, Q, S, q16, st, &launched); break;
      case 64: e = launch_fast<64, 16, 2>(xb, M, K, ldx, Q, S, q16, st, &launched); break;
      case 256: e = launch_fast<256, 16, 2>(xb, M, K, ldx, Q, S, q16, st, &launched); break;
      case 1024: e = launch_fast<1024, 64, 1>(xb, M, K, ldx, Q, S, q16, st, &launched); break;
      default: break;
    }
    if (e != cudaSuccess) return e;
    if (launched) {
      *path = 1;
      return cudaSuccess;
    }
  }
  const int threads = 256;
  const size_t smem = static_cast<size_t>(K) * sizeof(float);
  const long long grid = std::min<long long>(M, 64LL * device_sm_count());
  const float sdiv = scale_divisor(transform, G);
  if (in_dtype == CONVROT_DTYPE_BF16) {
    auto kern = rq_generic_kernel<__nv_bfloat16>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(static_cast<const __nv_bfloat16*>(X), M, K, ldx,
                                                             transform, G, signs, Q, S, q16, sdiv);
  } else {
    auto kern = rq_generic_kernel<float>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(static_cast<const float*>(X), M, K, ldx, transform, G,
                                                             signs, Q, S, q16, sdiv);
  }
  return cudaGetLastError();
}

}  // namespace convrot
