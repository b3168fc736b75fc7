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
// Register-resident kernel for bf16 input and the regular Hadamard.
//
// A CTA owns a tile of R consecutive rows and keeps all R*K values in
// registers, EPT per thread, across the row-absmax reduction.
//  Phase R: each thread takes SEGS segments of G1 consecutive elements,
//    loaded with 32-byte loads (a warp reads 1 KB contiguous per load), and
//    runs the radix-4 stages of the low digits in registers (G1 = 16: two
//    digits, G1 = 64: three).
//  Phase C (G > G1 only): the segments go through shared memory (fp32,
//    XOR-swizzled against bank conflicts) and come back as blocks of
//    G2 = G/G1 rows x 4 consecutive columns of the group viewed as a
//    G2 x G1 matrix; the high digits run in registers on those blocks.
//  Row absmax: shared-memory atomicMax per row.
//  Quantize: codes of 4 consecutive columns form one 32-bit word; they are
//    staged in shared memory (aliasing the fp32 buffer) and leave as 16-byte
//    coalesced stores. With G <= G1 each thread stores its segments directly.
// The loads of the next tile are issued before the output copy of the
// current one.

template <int G, int G1, int SEGS>
struct FastCfg {
  static constexpr int G2 = G > G1 ? G / G1 : 1;
  static constexpr int ND1 = ilog4_c(G < G1 ? G : G1);
  static constexpr int ND2 = ilog4_c(G2);
  static constexpr int EPT = SEGS * G1;
  static constexpr bool PHASE_C = G2 > 1;
  static constexpr int NB = PHASE_C ? EPT / (4 * G2) : 0;
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
// Staging buffers: word (4 codes) / 8-byte unit (4 fp16) index -> physical
// index; only bits >= 2 change, so aligned runs of 4 stay contiguous.
template <int G, int G1>
__device__ __forceinline__ int swz_word(int w) {
  constexpr int GS = ilog2_c(G / 4 > 1 ? G / 4 : 2);
  if constexpr (G1 == 16) {
    return w ^ (((w >> GS) & 7) << 2);
  } else {
    return w ^ (((w >> GS) & 1) << 4);
  }
}

template <int G, int G1, int SEGS>
__global__ void __launch_bounds__(384) rq_fast_kernel(const __nv_bfloat16* __restrict__ X, long long M, int K,
                                                       long long ldx, int R, int NT, int8_t* __restrict__ Q,
                                                       float* __restrict__ S, __half* __restrict__ Q16,
                                                       float s_div, int stage_bytes) {
  using C = FastCfg<G, G1, SEGS>;
  extern __shared__ __align__(128) unsigned char smem[];
  float* fbuf = reinterpret_cast<float*>(smem);
  uint32_t* stage_q = reinterpret_cast<uint32_t*>(smem);
  uint2* stage_h = reinterpret_cast<uint2*>(smem + stage_bytes);
  unsigned int* rowmax_buf = reinterpret_cast<unsigned int*>(smem + 4 * stage_bytes);  // [2][R]

  const int tid = threadIdx.x;
  const bool active = tid < NT;
  const long long ntiles = (M + R - 1) / R;
  const int tile_elems = R * K;

  // Static per-thread geometry: segment starts and phase-C block bases.
  int seg_off[SEGS];
#pragma unroll
  for (int j = 0; j < SEGS; ++j) seg_off[j] = (tid + j * NT) * G1;
  int blk_base[C::NB > 0 ? C::NB : 1];
  int blk_row[C::NB > 0 ? C::NB : 1];
  if constexpr (C::PHASE_C) {
    const int groups = K / G;
#pragma unroll
    for (int i = 0; i < C::NB; ++i) {
      const int b = tid + i * NT;
      const int c = b % (G1 / 4);
      const int rest = b / (G1 / 4);
      const int g = rest % groups;
      const int r = rest / groups;
      blk_row[i] = r;
      blk_base[i] = r * K + g * G + 4 * c;
    }
  }

  U32x8 raw[SEGS][C::LOADS];
  auto issue_loads = [&](long long tile) {
#pragma unroll
    for (int j = 0; j < SEGS; ++j) {
      const int e = seg_off[j];
      const int r = e / K, col = e % K;
      const long long row = tile * R + r;
      const bool ok = active && row < M;
      const __nv_bfloat16* p = X + row * ldx + col;
#pragma unroll
      for (int l = 0; l < C::LOADS; ++l) {
        if (ok) {
          raw[j][l] = ldg_nc_256(p + 16 * l);
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

    float v[C::EPT];
    // ---- phase R: widen, low-digit stages
#pragma unroll
    for (int j = 0; j < SEGS; ++j) {
#pragma unroll
      for (int l = 0; l < C::LOADS; ++l) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          v[j * G1 + l * 16 + 2 * k] = bf16lo_f32(raw[j][l].w[k]);
          v[j * G1 + l * 16 + 2 * k + 1] = bf16hi_f32(raw[j][l].w[k]);
        }
      }
    }
#pragma unroll
    for (int d = 0; d < C::ND1; ++d) {
      const int st = 1 << (2 * d);
#pragma unroll
      for (int j = 0; j < SEGS; ++j) {
#pragma unroll
        for (int base = 0; base < G1; base += 4 * st) {
#pragma unroll
          for (int o = 0; o < st; ++o) {
            float* p = v + j * G1 + base + o;
            h4_stage(p[0], p[st], p[2 * st], p[3 * st]);
          }
        }
      }
    }

    if constexpr (C::PHASE_C) {
      // ---- transpose through shared memory
      if (active) {
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
          const int c0 = seg_off[j] >> 2;
#pragma unroll
          for (int k = 0; k < G1 / 4; ++k) {
            float4 f = make_float4(v[j * G1 + 4 * k], v[j * G1 + 4 * k + 1], v[j * G1 + 4 * k + 2],
                                   v[j * G1 + 4 * k + 3]);
            reinterpret_cast<float4*>(fbuf)[swz_chunk<G, G1>(c0 + k)] = f;
          }
        }
      }
      __syncthreads();
      if (active) {
#pragma unroll
        for (int i = 0; i < C::NB; ++i) {
#pragma unroll
          for (int h = 0; h < C::G2; ++h) {
            const float4 f =
                reinterpret_cast<const float4*>(fbuf)[swz_chunk<G, G1>((blk_base[i] >> 2) + h * (G1 / 4))];
            float* p = v + i * 4 * C::G2 + 4 * h;
            p[0] = f.x;
            p[1] = f.y;
            p[2] = f.z;
            p[3] = f.w;
          }
        }
        // high-digit stages: digit d of h has stride 4^d rows = 4 * 4^d floats
#pragma unroll
        for (int d = 0; d < C::ND2; ++d) {
          const int st = 4 << (2 * d);
#pragma unroll
          for (int i = 0; i < C::NB; ++i) {
#pragma unroll
            for (int base = 0; base < 4 * C::G2; base += 4 * st) {
#pragma unroll
              for (int o = 0; o < st; o += 2) {
                float* p = v + i * 4 * C::G2 + base + o;
                float2 a0 = make_float2(p[0], p[1]), a1 = make_float2(p[st], p[st + 1]);
                float2 a2 = make_float2(p[2 * st], p[2 * st + 1]), a3 = make_float2(p[3 * st], p[3 * st + 1]);
                h4_stage(a0, a1, a2, a3);
                p[0] = a0.x; p[1] = a0.y;
                p[st] = a1.x; p[st + 1] = a1.y;
                p[2 * st] = a2.x; p[2 * st + 1] = a2.y;
                p[3 * st] = a3.x; p[3 * st + 1] = a3.y;
              }
            }
          }
        }
        // per-row absmax of each block
#pragma unroll
        for (int i = 0; i < C::NB; ++i) {
          float m = 0.0f;
#pragma unroll
          for (int e = 0; e < 4 * C::G2; e += 2)
            m = fmax3(m, fabsf(v[i * 4 * C::G2 + e]), fabsf(v[i * 4 * C::G2 + e + 1]));
          atomicMax(&rowmax[blk_row[i]], __float_as_uint(m));
        }
      }
    } else {
      if (active) {
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
          float m = 0.0f;
#pragma unroll
          for (int e = 0; e < G1; e += 2) m = fmax3(m, fabsf(v[j * G1 + e]), fabsf(v[j * G1 + e + 1]));
          atomicMax(&rowmax[seg_off[j] / K], __float_as_uint(m));
        }
      }
    }
    __syncthreads();

    // ---- quantize
    if (active) {
      if constexpr (C::PHASE_C) {
#pragma unroll
        for (int i = 0; i < C::NB; ++i) {
          const float amax = __uint_as_float(rowmax[blk_row[i]]);
          const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
#pragma unroll
          for (int h = 0; h < C::G2; ++h) {
            const float* p = v + i * 4 * C::G2 + 4 * h;
            const float t0 = fmaf(p[0], inv, kRoundMagic), t1 = fmaf(p[1], inv, kRoundMagic);
            const float t2 = fmaf(p[2], inv, kRoundMagic), t3 = fmaf(p[3], inv, kRoundMagic);
            const uint32_t b01 = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x0040);
            const uint32_t b23 = __byte_perm(__float_as_uint(t2), __float_as_uint(t3), 0x0040);
            const int w = (blk_base[i] >> 2) + h * (G1 / 4);
            stage_q[swz_word<G, G1>(w)] = __byte_perm(b01, b23, 0x5410);
            if (Q16) {
              const __half2 h01 = __floats2half2_rn(t0 - kRoundMagic, t1 - kRoundMagic);
              const __half2 h23 = __floats2half2_rn(t2 - kRoundMagic, t3 - kRoundMagic);
              uint2 u;
              u.x = *reinterpret_cast<const uint32_t*>(&h01);
              u.y = *reinterpret_cast<const uint32_t*>(&h23);
              stage_h[swz_word<G, G1>(w)] = u;
            }
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < SEGS; ++j) {
          const int e = seg_off[j];
          const int r = e / K, col = e % K;
          const long long row = tile * R + r;
          const float amax = __uint_as_float(rowmax[r]);
          const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
          uint32_t words[G1 / 4];
          uint32_t hw[G1 / 2];
#pragma unroll
          for (int k = 0; k < G1 / 4; ++k) {
            const float* p = v + j * G1 + 4 * k;
            const float t0 = fmaf(p[0], inv, kRoundMagic), t1 = fmaf(p[1], inv, kRoundMagic);
            const float t2 = fmaf(p[2], inv, kRoundMagic), t3 = fmaf(p[3], inv, kRoundMagic);
            const uint32_t b01 = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x0040);
            const uint32_t b23 = __byte_perm(__float_as_uint(t2), __float_as_uint(t3), 0x0040);
            words[k] = __byte_perm(b01, b23, 0x5410);
            if (Q16) {
              const __half2 h01 = __floats2half2_rn(t0 - kRoundMagic, t1 - kRoundMagic);
              const __half2 h23 = __floats2half2_rn(t2 - kRoundMagic, t3 - kRoundMagic);
              hw[2 * k] = *reinterpret_cast<const uint32_t*>(&h01);
              hw[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&h23);
            }
          }
          if (row < M) {
            int8_t* q = Q + row * (long long)K + col;
#pragma unroll
            for (int k = 0; k < G1 / 16; ++k)
              stg_128(q + 16 * k, make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]));
            if (Q16) {
              __half* qh = Q16 + row * (long long)K + col;
#pragma unroll
              for (int k = 0; k < G1 / 8; ++k)
                stg_128(qh + 8 * k, make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]));
            }
          }
        }
      }
    }
    for (int i = tid; i < R; i += blockDim.x)
      if (tile * R + i < M) S[tile * R + i] = __uint_as_float(rowmax[i]) / s_div;

    // ---- prefetch the next tile, then drain the staging buffers
    const long long next = tile + gridDim.x;
    if (next < ntiles) issue_loads(next);
    if constexpr (C::PHASE_C) {
      __syncthreads();
      const int pieces = tile_elems / 16;
      for (int pc = tid; pc < pieces; pc += blockDim.x) {
        const int e = pc * 16;
        const int r = e / K, col = e % K;
        const long long row = tile * R + r;
        if (row < M) {
          const uint4 val = reinterpret_cast<const uint4*>(stage_q)[swz_word<G, G1>(4 * pc) >> 2];
          stg_128(Q + row * (long long)K + col, val);
        }
      }
      if (Q16) {
        const int hpieces = tile_elems / 8;
        for (int pc = tid; pc < hpieces; pc += blockDim.x) {
          const int e = pc * 8;
          const int r = e / K, col = e % K;
          const long long row = tile * R + r;
          if (row < M) {
            const uint4 val = reinterpret_cast<const uint4*>(stage_h)[swz_word<G, G1>(2 * pc) >> 1];
            stg_128(Q16 + row * (long long)K + col, val);
          }
        }
      }
    }
    __syncthreads();
  }
}

// ================================================================ host =====

static float scale_divisor(int transform, int G) {
  if (transform == CONVROT_T_REGULAR_H4) return 127.0f * static_cast<float>(1 << (ilog2_c(G) / 2));
  if (transform == CONVROT_T_RHT) return static_cast<float>(127.0 * std::sqrt(static_cast<double>(G)));
  return 127.0f;
}

static int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
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
  const int tile_elems = R * K;
  // staging: int8 codes [tile] then fp16 copies [tile], each padded to 256 B;
  // the fp32 transpose buffer [tile] aliases both. rowmax follows.
  const int stage_bytes = ((tile_elems + 255) / 256) * 256;
  const int fbytes = ((tile_elems * 4 + 511) / 512) * 512;
  const int need = std::max(fbytes, 3 * stage_bytes);
  const int smem = std::max(need, 4 * stage_bytes) + 2 * R * 4;
  auto kern = rq_fast_kernel<G, G1, SEGS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaSuccess;
  const long long tiles = (M + R - 1) / R;
  const long long grid = std::min<long long>(tiles, static_cast<long long>(per_sm) * num_sms());
  kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(X, M, K, ldx, R, NT, Q, S, Q16,
                                                             scale_divisor(CONVROT_T_REGULAR_H4, G), stage_bytes);
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
      case 256: e = launch_fast<256, 16, 4>(xb, M, K, ldx, Q, S, q16, st, &launched); break;
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
  const long long grid = std::min<long long>(M, 64LL * num_sms());
  const float sdiv = scale_divisor(transform, G);
  if (in_dtype == CONVROT_DTYPE_BF16) {
    auto kern = rq_generic_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(static_cast<const __nv_bfloat16*>(X), M, K, ldx,
                                                             transform, G, signs, Q, S, q16, sdiv);
  } else {
    auto kern = rq_generic_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(static_cast<const float*>(X), M, K, ldx, transform, G,
                                                             signs, Q, S, q16, sdiv);
  }
  return cudaGetLastError();
}

}  // namespace convrot
