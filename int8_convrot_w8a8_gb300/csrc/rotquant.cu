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
//  * 4-bit codes ("feat: load ConvRot int4 and per-channel int8
//    safetensors", "Solution": values in [-7, 7], adjacent pairs in a byte)
//    use 7 in place of 127; they leave as two's-complement nibbles, element
//    2j in the low nibble of byte j, plus an e4m3 copy (every integer in
//    [-7, 7] is exact in e4m3) that the tensor cores read.
#include <algorithm>
#include <atomic>
#include <cstdio>

#include "common.cuh"

namespace convrot {

CONVROT_DEFINE_STATUS_WORD(status_word_rotquant)

// Eight magic-rounded values -> eight two's-complement nibbles, value i in
// bits 4i..4i+3 (the low bits of the rounded value are the code).
__device__ __forceinline__ uint32_t nibbles8(float t0, float t1, float t2, float t3, float t4, float t5, float t6,
                                             float t7) {
  const float t[8] = {t0, t1, t2, t3, t4, t5, t6, t7};
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) w |= (__float_as_uint(t[i]) & 0xFu) << (4 * i);
  return w;
}
// Two integer-valued floats -> two e4m3 bytes, the first in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

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

// qm = 127: Q int8 [M, K], Q16 fp16 copy; qm = 7: Q packed nibbles
// [M, K / 2], Q16 reinterpreted as the e4m3 copy [M, K] (bytes).
template <typename Tin>
__global__ void __launch_bounds__(256) rq_generic_kernel(const Tin* __restrict__ X, long long M, int K, long long ldx,
                                                         int transform, int G, const int8_t* __restrict__ signs,
                                                         int8_t* __restrict__ Q, float* __restrict__ S,
                                                         __half* __restrict__ Q16, float s_div, int qm) {
  asm volatile("griddepcontrol.launch_dependents;");  // see rq_lane_kernel
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
    const float inv = amax > 0.0f ? static_cast<float>(qm) / amax : 0.0f;
    if (qm == 127) {
      int8_t* q = Q ? Q + row * (long long)K : nullptr;
      for (int i = tid; i < K; i += nt) {
        const int c = code_from_magic(fmaf(buf[i], inv, kRoundMagic));
        if (q) q[i] = static_cast<int8_t>(c);
        if (Q16) Q16[row * (long long)K + i] = __int2half_rn(c);
      }
    } else {
      uint8_t* q4 = reinterpret_cast<uint8_t*>(Q) + row * (long long)(K / 2);
      uint8_t* f8 = Q16 ? reinterpret_cast<uint8_t*>(Q16) + row * (long long)K : nullptr;
      for (int j = tid; j < K / 2; j += nt) {
        const int c0 = code_from_magic(fmaf(buf[2 * j], inv, kRoundMagic));
        const int c1 = code_from_magic(fmaf(buf[2 * j + 1], inv, kRoundMagic));
        q4[j] = static_cast<uint8_t>((c0 & 0xF) | ((c1 & 0xF) << 4));
        if (f8) {
          const uint32_t b = e4m3x2(static_cast<float>(c0), static_cast<float>(c1));
          f8[2 * j] = static_cast<uint8_t>(b & 0xFF);
          f8[2 * j + 1] = static_cast<uint8_t>(b >> 8);
        }
      }
    }
    if (tid == 0) S[row] = amax / s_div;
    __syncthreads();
  }
}

// =============================================================== fast ======
// Fast kernel for bf16 input and the regular Hadamard (K a multiple of 64,
// G <= 1024).
//
// A CTA owns a tile of R consecutive rows (persistent grid-stride loop).
//  Load: one 3-D TMA copy per tile brings the R rows into shared memory as
//    128-byte lines (64 bf16) with the 128B swizzle; two stage buffers
//    alternate and the next tile's copy is issued when the current starts.
//  Each thread owns one line: 64 consecutive elements of a row, held in
//    registers as 32 fp32 pairs from load to store.
//  In-lane digits: the radix-4 stages of the three low digits (d0 scalar,
//    d1 and d2 on packed fp32x2 pairs of adjacent elements).
//  Digit 3 (G >= 256): the four lines of a group belong to the four lanes
//    of a quad; one fp32 transpose through shared memory inside the quad
//    (swizzled, conflict-free) turns the line index into a register index,
//    so the stage runs in registers on packed pairs.
//  Digit 4 (G = 1024): across the quads of a group with two shuffles per
//    element, u = x + x[a^1], w = x - x[a^1], y = u + w[a^2], which is the
//    same operation sequence, bit for bit, as the in-register stage.
//  Row absmax: warp reduction (one instruction when the warp lies in one
//    row), one shared-memory atomicMax per warp and row, one barrier.
//  Quantize straight from registers: codes leave as 32-byte stores (16-byte
//    after the quad transpose), fp16 copies as 32-byte stores: whole sectors.

// T: the transform; G: the group (regular Hadamard) or block (randomized
// Hadamard) size; the naive variant takes G = 1. XQ: the randomized
// Hadamard's cross-line stages through the quad transpose (rows of a
// multiple of 4 lines), else by shuffles.
template <int T, int G, bool XQ>
struct LaneCfg {
  static constexpr bool H4 = T == CONVROT_T_REGULAR_H4;
  static constexpr bool RHT = T == CONVROT_T_RHT;
  // regular Hadamard: radix-4 digits inside a 64-element line, then across lanes
  static constexpr int N = H4 ? ilog4_c(G) : 0;
  static constexpr int NIN = N < 3 ? N : 3;
  static constexpr int NX = N - NIN;
  // randomized Hadamard: radix-2 stages inside a line, then across lanes
  static constexpr int NB = RHT ? ilog2_c(G) : 0;
  static constexpr int NBIN = NB < 6 ? NB : 6;
  static constexpr int NBX = NB - NBIN;
  // line positions with distinct sign patterns (randomized Hadamard)
  static constexpr int NPOS = RHT && G > 64 ? G / 64 : 1;
  static_assert(NX <= 2 && NBX <= 2, "G <= 1024 (regular) or B <= 256 (randomized)");
  // the quad transpose runs: regular Hadamard digit 3, or the randomized
  // Hadamard's strides 64 and 128
  static constexpr bool QT = (H4 && NX >= 1) || (RHT && NBX >= 1 && XQ);
  // regular Hadamard: pair (v[2j], v[2j + 1]) holds elements (4j, 4j + 2) and
  // (4j + 1, 4j + 3), so digit 0 runs on packed pairs too; otherwise the pairs
  // hold (4j, 4j + 1) and (4j + 2, 4j + 3)
  static constexpr bool SPLIT = H4;
};

// Elements 4j .. 4j + 3, in order, from the pairs v[2j], v[2j + 1].
template <bool SPLIT>
__device__ __forceinline__ float4 elems4(float2 a, float2 b) {
  return SPLIT ? make_float4(a.x, b.x, a.y, b.y) : make_float4(a.x, a.y, b.x, b.y);
}

// One radix-2 Walsh-Hadamard stage across lanes (partner lane ^ MASK): the
// lower lane of the pair gets a + b, the upper one a - b (a the lower value),
// the same single roundings as the stage done in one place.
template <int MASK>
__device__ __forceinline__ float2 wht_xlane(float2 x, int lane) {
  float2 t;
  t.x = __shfl_xor_sync(0xffffffffu, x.x, MASK);
  t.y = __shfl_xor_sync(0xffffffffu, x.y, MASK);
  const float sg = (lane & MASK) ? -1.0f : 1.0f;
  return make_float2(fmaf(sg, x.x, t.x), fmaf(sg, x.y, t.y));
}

// One radix-4 stage, unnormalized, on lanes: this lane holds digit value
// a = (lane >> shift) & 3 of the quad it exchanges with.
template <int SHIFT>
__device__ __forceinline__ float2 h4_xlane(float2 x) {
  constexpr int m1 = 1 << SHIFT, m2 = 2 << SHIFT;
  float2 t;
  t.x = __shfl_xor_sync(0xffffffffu, x.x, m1);
  t.y = __shfl_xor_sync(0xffffffffu, x.y, m1);
  const float2 u = f2_add(x, t);
  float2 w = f2_sub(x, t);
  w.x = __shfl_xor_sync(0xffffffffu, w.x, m2);
  w.y = __shfl_xor_sync(0xffffffffu, w.y, m2);
  return f2_add(u, w);
}

template <int T, int G, int QM, bool XQ>
__global__ void __launch_bounds__(384) rq_lane_kernel(const __grid_constant__ CUtensorMap xmap, long long M, int K,
                                                       int R, int NT, const int8_t* __restrict__ signs,
                                                       int8_t* __restrict__ Q, float* __restrict__ S,
                                                       __half* __restrict__ Q16, float s_div, int stage_bytes,
                                                       int tbytes, int box_lines, long long spin_limit) {
  using C = LaneCfg<T, G, XQ>;
  // a programmatic dependent launch (the GEMM) may be scheduled now; it
  // waits for this grid to complete before it reads the codes
  asm volatile("griddepcontrol.launch_dependents;");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage_base = smem_u32(smem);
  const uint32_t tbuf = stage_base + 2 * stage_bytes;  // fp32 quad-transpose buffer (G >= 256)
  unsigned int* rowmax_buf = reinterpret_cast<unsigned int*>(smem + 2 * stage_bytes + tbytes);  // [3][R]
  uint64_t* bar = reinterpret_cast<uint64_t*>(rowmax_buf + ((3 * R + 1) & ~1));         // [2]
  // randomized Hadamard: per line position, 32 words that flip the sign bits
  // of the packed bf16 pairs (bit 15: element 2k, bit 31: element 2k + 1)
  uint32_t* sign_tab =
      reinterpret_cast<uint32_t*>((reinterpret_cast<uintptr_t>(bar + 2) + 15) & ~uintptr_t(15));  // [NPOS][32]

  const int tid = threadIdx.x, lane = tid & 31;
  const bool active = tid < NT;
  const long long ntiles = (M + R - 1) / R;
  const int lines_per_row = K >> 6;
  const int my_row = active ? tid / lines_per_row : -1;
  const uint32_t tile_bytes = static_cast<uint32_t>(R) * static_cast<uint32_t>(K) * 2u;
  const long long total_elems = M * static_cast<long long>(K);
  // whether this warp's active lanes all belong to one row
  const int row_first = __shfl_sync(0xffffffffu, my_row, 0);
  const bool warp_one_row = __all_sync(0xffffffffu, my_row == row_first);

  // Quad transpose (regular Hadamard G >= 256, randomized Hadamard B >= 128
  // on rows of 4k lines): the 4 lanes of a quad own 4 consecutive lines. Each
  // writes its line (fp32, 16 chunks of 16 bytes) and reads back the
  // 16-element run at offset 16a (a = lane & 3) of all 4 lines, so the line
  // index becomes a register index. Chunk c of line l sits at chunk
  // c ^ (bitrev3(l mod 8) ^ ((c >> 3) << 1)) of its 256-byte slot:
  // conflict-free for the line writes and for the transposed reads.
  const int qa = tid & 3;
  uint32_t t_wr = 0;      // write base, XOR-ed with the compile-time part of the swizzle
  uint32_t t_rd[4] = {};  // read base of line (tid & ~3) + r, XOR-ed likewise
  if constexpr (C::QT) {
    auto bitrev3 = [](int x) { return ((x & 1) << 2) | (x & 2) | ((x >> 2) & 1); };
    t_wr = (tbuf + (static_cast<uint32_t>(tid) << 8)) | (static_cast<uint32_t>(bitrev3(tid & 7)) << 4);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int l = (tid & ~3) + r;
      const int tr = (4 * qa) ^ bitrev3(l & 7) ^ ((qa >> 1) << 1);
      t_rd[r] = (tbuf + (static_cast<uint32_t>(l) << 8)) | (static_cast<uint32_t>(tr) << 4);
    }
  }

  long long tile = blockIdx.x;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the first tile's copy is in flight during the set-up below
    if (tile < ntiles) {
      mbar_expect_tx(&bar[0], tile_bytes);
      for (int l0 = 0; l0 < lines_per_row; l0 += box_lines)
        tma_load_3d(stage_base + l0 * 128, &xmap, 0, l0, static_cast<int>(tile * R), &bar[0]);
    }
  }
  // Row maxima cycle through three buffers. Iteration `it` uses buffer
  // it % 3 and clears (it + 1) % 3, last used two iterations earlier: every
  // thread has passed the barrier of iteration it - 1, so every thread has
  // finished reading it.
  for (int i = tid; i < 3 * R; i += blockDim.x) rowmax_buf[i] = 0u;
  // the slots of threads past NT (padding to whole warps) never receive a
  // line: they hold zeros, so every thread loads its slot unconditionally
  for (int i = NT * 8 + tid; i < static_cast<int>(blockDim.x) * 8; i += blockDim.x) {
    const uint32_t z = 0u;
    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(stage_base + 16u * i), "r"(z) : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(stage_base + stage_bytes + 16u * i), "r"(z)
                 : "memory");
  }
  if constexpr (C::RHT) {
    for (int i = tid; i < C::NPOS * 32; i += blockDim.x) {
      const int e = ((i >> 5) * 64 + 2 * (i & 31)) & (G - 1);  // element of the block
      sign_tab[i] = (signs[e] < 0 ? 0x8000u : 0u) | (signs[(e + 1) & (G - 1)] < 0 ? 0x80000000u : 0u);
    }
  }
  __syncthreads();
  // the line position of this thread in its block (its lines are fixed)
  const uint32_t my_signs = smem_u32(sign_tab) + static_cast<uint32_t>(((tid % lines_per_row) % C::NPOS) * 128);

  for (int it = 0; tile < ntiles; tile += gridDim.x, ++it) {
    const int buf = it & 1;
    unsigned int* rowmax = rowmax_buf + (it % 3) * R;
    for (int i = tid; i < R; i += blockDim.x) rowmax_buf[((it + 1) % 3) * R + i] = 0u;
    const long long next = tile + gridDim.x;
    // the other stage buffer was last read before the previous iteration's
    // barrier: refill it with the next tile now
    if (tid == 0 && next < ntiles) {
      mbar_expect_tx(&bar[buf ^ 1], tile_bytes);
      for (int l0 = 0; l0 < lines_per_row; l0 += box_lines)
        tma_load_3d(stage_base + (buf ^ 1) * stage_bytes + l0 * 128, &xmap, 0, l0, static_cast<int>(next * R),
                    &bar[buf ^ 1]);
    }
    if (!mbar_wait_bounded(&bar[buf], (it >> 1) & 1, spin_limit) && tid == 0) record_status(CONVROT_ERR_TIMEOUT);

    // ---- this thread's line: 64 bf16 -> 32 fp32 pairs
    float2 v[32];
    {
      const uint32_t lb = stage_base + buf * stage_bytes + (static_cast<uint32_t>(tid) << 7);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        // every thread has a slot; the slots of threads past NT hold zeros
        uint32_t w0, w1, w2, w3;
        const uint32_t addr = lb + ((k ^ (tid & 7)) << 4);
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(addr));
        if constexpr (C::RHT) {
          uint32_t m0, m1, m2, m3;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(m0), "=r"(m1), "=r"(m2), "=r"(m3)
                       : "r"(my_signs + 16 * k));
          w0 ^= m0;
          w1 ^= m1;
          w2 ^= m2;
          w3 ^= m3;
        }
        if constexpr (C::SPLIT) {
          v[4 * k + 0] = make_float2(bf16lo_f32(w0), bf16lo_f32(w1));
          v[4 * k + 1] = make_float2(bf16hi_f32(w0), bf16hi_f32(w1));
          v[4 * k + 2] = make_float2(bf16lo_f32(w2), bf16lo_f32(w3));
          v[4 * k + 3] = make_float2(bf16hi_f32(w2), bf16hi_f32(w3));
        } else {
          v[4 * k + 0] = make_float2(bf16lo_f32(w0), bf16hi_f32(w0));
          v[4 * k + 1] = make_float2(bf16lo_f32(w1), bf16hi_f32(w1));
          v[4 * k + 2] = make_float2(bf16lo_f32(w2), bf16hi_f32(w2));
          v[4 * k + 3] = make_float2(bf16lo_f32(w3), bf16hi_f32(w3));
        }
      }
    }
    // ---- digit 0 on elements 4q .. 4q+3, held as v[2q] = (x0, x2), v[2q+1] =
    // (x1, x3): u = (x0 + x1, x2 + x3), w = (x0 - x1, x2 - x3), then
    // (x0', x2') = u + (w2, w0) and (x1', x3') = u - (w2, w0), the same single
    // roundings as the scalar stage
    if constexpr (C::NIN >= 1) {
      static_assert(C::SPLIT, "the regular Hadamard keeps split pairs");
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float2 u = f2_add(v[2 * q], v[2 * q + 1]);
        const float2 w = f2_sub(v[2 * q], v[2 * q + 1]);
        const float2 ws = make_float2(w.y, w.x);
        v[2 * q] = f2_add(u, ws);
        v[2 * q + 1] = f2_sub(u, ws);
      }
    }
    // ---- digit 1 (stride 4 elements = 2 pairs) and digit 2 (stride 16 = 8 pairs), packed
    if constexpr (C::NIN >= 2) {
#pragma unroll
      for (int b = 0; b < 32; b += 8)
#pragma unroll
        for (int o = 0; o < 2; ++o) h4_stage(v[b + o], v[b + o + 2], v[b + o + 4], v[b + o + 6]);
    }
    if constexpr (C::NIN >= 3) {
#pragma unroll
      for (int o = 0; o < 8; ++o) h4_stage(v[o], v[o + 8], v[o + 16], v[o + 24]);
    }
    // after the quad transpose v[8r + i] holds elements 16a + 2i, +1 of line
    // (tid & ~3) + r
    auto quad_transpose = [&]() {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint32_t addr = t_wr ^ (static_cast<uint32_t>(k ^ ((k >> 3) << 1)) << 4);
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v[2 * k].x), "f"(v[2 * k].y),
                     "f"(v[2 * k + 1].x), "f"(v[2 * k + 1].y)
                     : "memory");
      }
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float4 f;
          asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                       : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                       : "r"(t_rd[r] ^ (static_cast<uint32_t>(c) << 4))
                       : "memory");
          v[8 * r + 2 * c] = make_float2(f.x, f.y);
          v[8 * r + 2 * c + 1] = make_float2(f.z, f.w);
        }
    };
    // ---- digit 3 through the quad transpose, then in registers
    if constexpr (C::H4 && C::NX >= 1) {
      quad_transpose();
#pragma unroll
      for (int i = 0; i < 8; ++i) h4_stage(v[i], v[8 + i], v[16 + i], v[24 + i]);
    }
    // ---- digit 4 (G = 1024): across the 4 quads of a group, lane bits 2-3
    if constexpr (C::NX >= 2) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = h4_xlane<2>(v[i]);
    }

    // ---- randomized Hadamard: radix-2 stages, stride 1 first (in the pair),
    // strides 2..32 across pairs (packed), 64 and 128 across lanes
    if constexpr (C::NBIN >= 1) {
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const float a = v[q].x, b = v[q].y;
        v[q] = make_float2(a + b, a - b);
      }
    }
#pragma unroll
    for (int st = 1; st < 6; ++st) {
      if (st < C::NBIN) {
        const int d = 1 << (st - 1);  // pair distance
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          if ((q & d) == 0) {
            const float2 a = v[q], b = v[q + d];
            v[q] = f2_add(a, b);
            v[q + d] = f2_sub(a, b);
          }
        }
      }
    }
    if constexpr (C::RHT && C::QT) {
      // strides 64 and 128 (lines r ^ 1, r ^ 2) in registers after the transpose
      quad_transpose();
#pragma unroll
      for (int r = 0; r < 4; r += 2)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 a = v[8 * r + i], b = v[8 * (r + 1) + i];
          v[8 * r + i] = f2_add(a, b);
          v[8 * (r + 1) + i] = f2_sub(a, b);
        }
      if constexpr (C::NBX >= 2) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 a = v[8 * r + i], b = v[8 * (r + 2) + i];
            v[8 * r + i] = f2_add(a, b);
            v[8 * (r + 2) + i] = f2_sub(a, b);
          }
      }
    } else {
      if constexpr (C::NBX >= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = wht_xlane<1>(v[i], lane);
      }
      if constexpr (C::NBX >= 2) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = wht_xlane<2>(v[i], lane);
      }
    }

    // ---- row absmax
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = fmax3(m, fabsf(v[i].x), fabsf(v[i].y));
    if (warp_one_row) {
      const unsigned mx = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      if (lane == 0 && row_first >= 0) atomicMax(&rowmax[row_first], mx);
    } else {
      const unsigned grp = __match_any_sync(0xffffffffu, my_row);
      const unsigned mx = __reduce_max_sync(grp, __float_as_uint(m));
      if (active && lane == __ffs(grp) - 1) atomicMax(&rowmax[my_row], mx);
    }
    __syncthreads();

    // ---- quantize and store
    if (active && QM == 7) {
      // 4-bit: 16 values -> 8 bytes of nibbles and 16 e4m3 bytes
      const float amax = __uint_as_float(rowmax[my_row]);
      const float inv = amax > 0.0f ? 7.0f / amax : 0.0f;
      const float2 inv2 = make_float2(inv, inv);
      const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
      const long long tile_e = (tile * R) * static_cast<long long>(K);
      uint8_t* q4 = reinterpret_cast<uint8_t*>(Q);
      uint8_t* f8 = reinterpret_cast<uint8_t*>(Q16);
      auto emit16_w4 = [&](int p0, long long e) {
        float2 t[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = f2_fma(v[p0 + k], inv2, mg2);
        const float4 f0 = elems4<C::SPLIT>(t[0], t[1]), f1 = elems4<C::SPLIT>(t[2], t[3]);
        const float4 f2 = elems4<C::SPLIT>(t[4], t[5]), f3 = elems4<C::SPLIT>(t[6], t[7]);
        const uint32_t n0 = nibbles8(f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w);
        const uint32_t n1 = nibbles8(f2.x, f2.y, f2.z, f2.w, f3.x, f3.y, f3.z, f3.w);
        asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(q4 + (e >> 1)), "r"(n0), "r"(n1) : "memory");
        if (f8) {
          uint32_t fw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 c = elems4<C::SPLIT>(f2_sub(t[2 * k], mg2), f2_sub(t[2 * k + 1], mg2));
            fw[k] = e4m3x2(c.x, c.y) | (e4m3x2(c.z, c.w) << 16);
          }
          stg_128(f8 + e, make_uint4(fw[0], fw[1], fw[2], fw[3]));
        }
      };
      if (tile_e + (static_cast<long long>(tid) << 6) < total_elems) {
        if constexpr (C::QT) {
#pragma unroll
          for (int r = 0; r < 4; ++r)
            emit16_w4(8 * r, tile_e + (static_cast<long long>((tid & ~3) + r) << 6) + 16 * qa);
        } else {
          const long long e0 = tile_e + (static_cast<long long>(tid) << 6);
#pragma unroll
          for (int h = 0; h < 4; ++h) emit16_w4(8 * h, e0 + 16 * h);
        }
      }
    } else if (active) {
      const float amax = __uint_as_float(rowmax[my_row]);
      const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
      const float2 inv2 = make_float2(inv, inv);
      const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
      const long long tile_e = (tile * R) * static_cast<long long>(K);
      // 16 values -> 16 codes (one 16-byte store) and 16 fp16 copies (one 32-byte store)
      auto emit16 = [&](int p0, long long e) {
        uint32_t words[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 ta = f2_fma(v[p0 + 2 * k], inv2, mg2);
          const float2 tb = f2_fma(v[p0 + 2 * k + 1], inv2, mg2);
          const float4 t = elems4<C::SPLIT>(ta, tb);  // elements 4k .. 4k+3 of the run
          const uint32_t b01 = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x0040);
          const uint32_t b23 = __byte_perm(__float_as_uint(t.z), __float_as_uint(t.w), 0x0040);
          words[k] = __byte_perm(b01, b23, 0x5410);
          if (Q16) {  // reuse the rounded values: code = t - magic, exact in fp16
            v[p0 + 2 * k] = f2_sub(ta, mg2);
            v[p0 + 2 * k + 1] = f2_sub(tb, mg2);
          }
        }
        if (Q) stg_128(Q + e, make_uint4(words[0], words[1], words[2], words[3]));
        if (Q16) {
          uint32_t hw[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 c = elems4<C::SPLIT>(v[p0 + 2 * k], v[p0 + 2 * k + 1]);
            const __half2 p = __floats2half2_rn(c.x, c.y), p2 = __floats2half2_rn(c.z, c.w);
            hw[2 * k] = *reinterpret_cast<const uint32_t*>(&p);
            hw[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&p2);
          }
          stg_256(Q16 + e, hw);
        }
      };
      if (tile_e + (static_cast<long long>(tid) << 6) < total_elems) {
        if constexpr (C::QT) {
#pragma unroll
          for (int r = 0; r < 4; ++r)
            emit16(8 * r, tile_e + (static_cast<long long>((tid & ~3) + r) << 6) + 16 * qa);
        } else {
          // the whole line: codes as two 32-byte stores, fp16 copies as four
          const long long e0 = tile_e + (static_cast<long long>(tid) << 6);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t words[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 ta = f2_fma(v[16 * h + 2 * k], inv2, mg2);
              const float2 tb = f2_fma(v[16 * h + 2 * k + 1], inv2, mg2);
              const float4 t = elems4<C::SPLIT>(ta, tb);
              const uint32_t b01 = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x0040);
              const uint32_t b23 = __byte_perm(__float_as_uint(t.z), __float_as_uint(t.w), 0x0040);
              words[k] = __byte_perm(b01, b23, 0x5410);
              if (Q16) {
                v[16 * h + 2 * k] = f2_sub(ta, mg2);
                v[16 * h + 2 * k + 1] = f2_sub(tb, mg2);
              }
            }
            if (Q) stg_256(Q + e0 + 32 * h, words);
          }
          if (Q16) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              uint32_t hw[8];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 c = elems4<C::SPLIT>(v[8 * h + 2 * k], v[8 * h + 2 * k + 1]);
                const __half2 p = __floats2half2_rn(c.x, c.y), p2 = __floats2half2_rn(c.z, c.w);
                hw[2 * k] = *reinterpret_cast<const uint32_t*>(&p);
                hw[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&p2);
              }
              stg_256(Q16 + e0 + 16 * h, hw);
            }
          }
        }
      }
    }
    for (int i = tid; i < R; i += blockDim.x)
      if (tile * R + i < M) S[tile * R + i] = __uint_as_float(rowmax[i]) / s_div;
  }
}

// ========================================================== tensor-core ===
// Regular Hadamard (G = 4 .. 1024, K a multiple of 256) with the two lowest
// radix-4 digits, the 16-point stage, on the tensor cores: mma.sync m16n8k16
// bf16 -> fp32 straight from the TMA-staged tile, against the unnormalized
// +-1 matrix of that stage (exact in bf16; the products are exact and the
// tensor core sums 16 of them in fp32). The digits above it run on fp32
// registers, as in the register kernel, and the codes and scales follow the
// same arithmetic (one division per row, one rounding per code).
//
// Work split. Every 256 consecutive values of a row form a superblock of 16
// chunks of 16 values. A warp owns 8 consecutive superblocks of the tile;
// the thread with MMA group id g = lane / 4 owns superblock g of its warp,
// and in it positions 4t .. 4t + 3 (t = lane % 4) of all 16 chunks: the 64
// values that the digits above the chunk combine.
//  * A operand: 8 MMA tiles of 16 rows. Row g + 8h of tile u is chunk
//    (2u + h) ^ g of superblock g, so every thread group meets each of its
//    chunks once, and the XOR spreads the eight rows one ldmatrix phase
//    reads over distinct 16-byte bank groups of the 128B-swizzled stage (the
//    superblock's first line is 4 x its index, so the swizzle phase of each
//    row is known on the host; the same holds for the int8 stores).
//  * B operand: the 16 x 16 matrix with its output columns permuted so that
//    the thread's four result columns are positions 4t .. 4t + 3 (n-block 0:
//    4t, 4t + 1; n-block 1: 4t + 2, 4t + 3).
//  * Results: slot s = 2u + h holds chunk s ^ g. The radix-4 stage is
//    unchanged when all four digit values are XOR-ed with one constant (its
//    -1 sits where b = a ^ 3), so the digits above the chunk run on slots,
//    with compile-time register indices; across lanes (G = 1024) a partner's
//    matching chunk sits in its slot s ^ (g ^ g_partner).
//  * Row maximum, quantization and stores as in the register kernel; the
//    codes leave as 4-byte words (4 consecutive codes), the fp16 copy as
//    8-byte pieces.
// Pipeline: persistent CTAs, a ring of STAGES TMA stages (3-D box of R
// rows as 128-byte lines, 128B swizzle), each refilled with the tile STAGES
// iterations ahead as soon as every warp has passed the row-max barrier.

// Entry (p, k) of the unnormalized 16-point stage: the Kronecker square of
// 2*H4 (entries +-1, -1 where the two digits satisfy b = a ^ 3), or for
// G = 4 the block-diagonal I4 (x) 2*H4.
__host__ __device__ constexpr float h16_entry(int G, int p, int k) {
  const float lo = ((p & 3) ^ (k & 3)) == 3 ? -1.0f : 1.0f;
  if (G == 4) return (p >> 2) == (k >> 2) ? lo : 0.0f;
  return (((p >> 2) ^ (k >> 2)) == 3 ? -1.0f : 1.0f) * lo;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

constexpr int kMmaMaxWarps = 12;
constexpr int kMmaMinWarps = 6;

// Dynamic tile hand-out of the tensor-core kernel. Static round-robin tiles
// leave the GPU waiting on its slowest CTAs (on GB300 the CTAs of one launch,
// each with the same tile count, finish up to 25 % apart). Instead every CTA
// claims its next tile from a counter; one counter pair (tiles claimed, CTAs
// done) per launch slot, zero when the module loads; the last CTA of a launch
// to finish puts its pair back to zero. Launches take the slots in turn, so
// up to kRqSchedSlots launches may be in flight on a device at once.
constexpr int kRqSchedSlots = 256;
static __device__ unsigned int g_rq_sched[kRqSchedSlots][2];

// What a launch computes. kRqFull: codes and scales (the row maximum taken
// over the given columns). kRqAbsmax: only the row maxima of the rotated
// slice, max_i |X_rot[r, i]|, into amax. kRqGivenMax: codes and scales with
// the row maxima read from amax (taken over a whole row whose columns are
// split over several calls, as in a row-parallel linear).
constexpr int kRqFull = 0, kRqAbsmax = 1, kRqGivenMax = 2;

// QM = 127: WQ / WH write the int8 codes / their fp16 copy. QM = 7 (4-bit
// codes in [-7, 7]): WQ writes the packed nibbles (element 2j in the low
// nibble of byte j), WH their e4m3 copy.
// NB: staging buffers for the outputs. With two, a tile's bulk store is
// issued after the next tile's row-max barrier, so a tile costs one CTA-wide
// barrier instead of two.
template <int G, int STAGES, bool WQ, bool WH, int MODE, int QM, int NB, bool RAG>
__global__ void __launch_bounds__(32 * kMmaMaxWarps) rq_mma_kernel(
    const __grid_constant__ CUtensorMap xmap, long long M, int K, int R, int nsb, int8_t* __restrict__ Q,
    float* __restrict__ S, __half* __restrict__ Q16, float* __restrict__ amax, float s_div, int stage_bytes,
    int box_lines, int slot, long long spin_limit) {
  static_assert(MODE != kRqAbsmax || (!WQ && !WH), "the row-max mode writes no codes");
  // RAG: K a multiple of 64 but not of 256, so a superblock (4 lines) may
  // end in the next row of the tile; its groups (G <= 64) stay within a line
  static_assert(!RAG || (G <= 64 && MODE == kRqFull), "superblocks across rows: G <= 64, codes and scales");
  // the normalization 2^-n of R_G is a power of two: scaling a maximum by it
  // (or back) is exact
  constexpr float kNorm = 1.0f / static_cast<float>(1 << ilog4_c(G));
  static_assert(G == 4 || G == 16 || G == 64 || G == 256 || G == 1024, "regular Hadamard group");
  asm volatile("griddepcontrol.launch_dependents;");  // see rq_lane_kernel
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage_base = smem_u32(smem);
  // output staging: the tile's tensor-core copy [R, K] (fp16, or e4m3 for
  // 4-bit codes) and its codes [R, K] (int8, or nibbles [R, K / 2]); each
  // present when asked for, each starting on a 128-byte boundary, each
  // written out by one bulk copy per tile
  constexpr uint32_t kHB2 = QM == 127 ? 4 : 2;  // bytes per element of the copy, x2
  constexpr uint32_t kQB2 = QM == 127 ? 2 : 1;  // bytes per element of the codes, x2
  const uint32_t tile_elems = static_cast<uint32_t>(R) * static_cast<uint32_t>(K);
  const uint32_t h_bytes = WH ? kHB2 * tile_elems / 2 : 0u, q_bytes = WQ ? kQB2 * tile_elems / 2 : 0u;
  const uint32_t buf_bytes = (h_bytes + q_bytes + 1023u) & ~1023u;  // one staging buffer, 1 KB aligned
  const uint32_t out_h = stage_base + STAGES * stage_bytes;
  const uint32_t out_q = out_h + h_bytes;
  unsigned int* rowmax_buf =
      reinterpret_cast<unsigned int*>(smem + STAGES * stage_bytes + NB * buf_bytes);  // [3][R]
  uint64_t* full = reinterpret_cast<uint64_t*>(rowmax_buf + ((3 * R + 1) & ~1));            // [STAGES]
  long long* stage_tile = reinterpret_cast<long long*>(full + STAGES);                      // [STAGES]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long ntiles = (M + R - 1) / R;
  const int lines_per_row = K >> 6;
  const int sb_per_row = K >> 8;
  const uint32_t tile_bytes = static_cast<uint32_t>(R) * static_cast<uint32_t>(K) * 2u;

  // Tiles: the first STAGES rounds go out round-robin (tile blockIdx.x +
  // k * gridDim.x for the k-th stage filled), the rest by claims on the
  // counter, numbered from STAGES * gridDim.x. Only tid 0 claims, one claim
  // ahead (the atomic's round trip overlaps a whole tile). Tiles come out in
  // increasing order for each CTA, so once one lies past the end every later
  // one does too, and a CTA leaves with no copy in flight.
  unsigned int* claims = &g_rq_sched[slot][0];
  const long long dyn_base = static_cast<long long>(STAGES) * gridDim.x;
  unsigned int pending = 0;  // tid 0: the claim for the next refill
  bool exhausted = false;    // tid 0: a claim came back past the end
  auto fill = [&](int s, long long c) {  // tid 0: start stage s on tile c (or mark it empty)
    if (c < ntiles) {
      stage_tile[s] = c;
      mbar_expect_tx(&full[s], tile_bytes);
      for (int l0 = 0; l0 < lines_per_row; l0 += box_lines)
        tma_load_3d(stage_base + s * stage_bytes + l0 * 128, &xmap, 0, l0, static_cast<int>(c * R), &full[s]);
    } else {
      exhausted = true;
      stage_tile[s] = -1;
      mbar_arrive(&full[s]);
    }
  };
  // (tid 0) bulk-stores tile tl's codes from staging buffer b
  auto store_tile = [&](long long tl, int b) {
    const long long rows = M - tl * R < R ? M - tl * R : R;
    const long long e0 = tl * R * static_cast<long long>(K);
    const uint32_t n = static_cast<uint32_t>(rows * K);
    const uint32_t off = static_cast<uint32_t>(b) * buf_bytes;
    if constexpr (WQ)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       reinterpret_cast<unsigned char*>(Q) + e0 * kQB2 / 2),
                   "r"(out_q + off), "r"(kQB2 * n / 2)
                   : "memory");
    if constexpr (WH)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       reinterpret_cast<unsigned char*>(Q16) + e0 * kHB2 / 2),
                   "r"(out_h + off), "r"(kHB2 * n / 2)
                   : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  };
  // the first tile's copy starts before anything else, alone: the first
  // tiles of all CTAs then reach the SMs ahead of the deeper stages
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fill(0, blockIdx.x);
  }

  // ---- result side: this thread's superblock and positions
  const int g = lane >> 2, t = lane & 3;
  const int sb = warp * 8 + g;
  const bool sb_valid = sb < nsb;
  // row within the tile (of the superblock's first line)
  const int my_row = sb_valid ? (RAG ? 4 * sb / lines_per_row : sb / sb_per_row) : -1;
  // RAG: the row of the superblock's last line, and bit h set where slots
  // 4h .. 4h + 3 (line h ^ (g >> 2) of the superblock) lie in that row but
  // not in my_row
  int my_row2 = my_row;
  unsigned in2 = 0u;
  if constexpr (RAG) {
    if (sb_valid) {
      my_row2 = (4 * sb + 3) / lines_per_row;
#pragma unroll
      for (int h = 0; h < 4; ++h)
        if ((4 * sb + (h ^ (g >> 2))) / lines_per_row != my_row) in2 |= 1u << h;
    }
  }
  // staging address of positions 4t .. 4t + 3 of chunk g of this superblock
  // (the superblocks of a tile are consecutive in the dense output); chunk
  // s ^ g is then at that address XOR (chunk bytes) * s, since the chunk
  // offset bits of the superblock's base are zero.
  // G = 1024: after the digit-4 exchange below, slot s of the lane with
  // j = g & 3 holds chunk ((s & 12) ^ 4 (g >> 2)) | j of superblock
  // 4 (g >> 2) + (j ^ (s & 3)) of the warp's group; its offset from the
  // tile's staging base is my_q XOR a constant of s (the group's base is a
  // multiple of the group's bytes, so the fields do not carry).
  const int g2 = g >> 2, jq = g & 3;
  const uint32_t my_q =
      G == 1024 ? 128u * kQB2 * static_cast<uint32_t>(warp * 8 + 4 * g2 + jq) + 8u * kQB2 * (4 * g2 + jq) + 2u * kQB2 * t
                : (out_q + static_cast<uint32_t>(sb) * 128u * kQB2 + 2u * kQB2 * t) | (8u * kQB2 * g);
  const uint32_t my_h =
      G == 1024 ? 128u * kHB2 * static_cast<uint32_t>(warp * 8 + 4 * g2 + jq) + 8u * kHB2 * (4 * g2 + jq) + 2u * kHB2 * t
                : (out_h + static_cast<uint32_t>(sb) * 128u * kHB2 + 2u * kHB2 * t) | (8u * kHB2 * g);
  // staging address of slot s (buffer offset bsel added by the caller)
  auto q_at = [&](int s) -> uint32_t {
    if constexpr (G == 1024) return out_q + (my_q ^ (128u * kQB2 * (s & 3) + 8u * kQB2 * (s & 12)));
    return my_q ^ (8u * kQB2 * s);
  };
  auto h_at = [&](int s) -> uint32_t {
    if constexpr (G == 1024) return out_h + (my_h ^ (128u * kHB2 * (s & 3) + 8u * kHB2 * (s & 12)));
    return my_h ^ (8u * kHB2 * s);
  };

  // ---- operand side: the rows this lane addresses for ldmatrix.x4
  // (matrix m = lane / 8: h = m & 1 picks row g + 8h, hf = m >> 1 the 8-value
  // half of the chunk; the row's superblock is that of group lane % 8)
  uint32_t a_off[8];
  {
    const int ga = lane & 7, h = (lane >> 3) & 1, hf = lane >> 4;
    int sba = warp * 8 + ga;
    if (sba >= nsb) sba = ga < nsb ? ga : 0;  // padding groups read real data; their results are dropped
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = (2 * u + h) ^ ga;
      const int L = 4 * sba + (j >> 2);
      const int c = (2 * (j & 3) + hf) ^ (L & 7);
      a_off[u] = static_cast<uint32_t>(L * 128 + c * 16);
    }
  }
  // ---- B fragments of the two n-blocks: b0 = rows k = 2t, 2t + 1 and b1 =
  // rows 2t + 8, 2t + 9 of column n = g, which is position 4(g / 2) + 2nb + g % 2
  uint32_t bfrag[2][2];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) {
    const int p = 4 * (g >> 1) + 2 * nb + (g & 1);
    bfrag[nb][0] = bf16x2_bits(h16_entry(G, p, 2 * t), h16_entry(G, p, 2 * t + 1));
    bfrag[nb][1] = bf16x2_bits(h16_entry(G, p, 2 * t + 8), h16_entry(G, p, 2 * t + 9));
  }

  for (int i = tid; i < 3 * R; i += blockDim.x) rowmax_buf[i] = 0u;
  __syncthreads();
  // the deeper stages of the first round-robin rounds, then the first claim
  if (tid == 0) {
    for (int s = 1; s < STAGES; ++s) fill(s, blockIdx.x + static_cast<long long>(s) * gridDim.x);
    if (!exhausted) pending = atomicAdd(claims, 1u);
  }

  const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
  long long prev_tile = -1;  // NB = 2: the tile whose codes wait in the other staging buffer
  int prev_it = 0;           //        and the iteration that wrote them
  for (int it = 0;; ++it) {
    const int st = it % STAGES;
    unsigned int* rowmax = rowmax_buf + (it % 3) * R;
    for (int i = tid; i < R; i += blockDim.x) rowmax_buf[((it + 1) % 3) * R + i] = 0u;
    if (!mbar_wait_bounded(&full[st], (it / STAGES) & 1, spin_limit) && tid == 0) record_status(CONVROT_ERR_TIMEOUT);
    // the stage's tile (written by tid 0 before its barrier phase completed)
    const long long tile = *reinterpret_cast<volatile long long*>(&stage_tile[st]);
    if (tile < 0) break;

    // ---- 16-point stage on the tensor cores: v[s][nb] = positions
    // (4t + 2nb, 4t + 2nb + 1) of the chunk in slot s
    float2 v[16][2];
    const uint32_t sbase = stage_base + st * stage_bytes;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint32_t a0, a1, a2, a3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                   : "r"(sbase + a_off[u]));
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        float d[4];
        mma_bf16_16816(d, a0, a1, a2, a3, bfrag[nb][0], bfrag[nb][1]);
        v[2 * u][nb] = make_float2(d[0], d[1]);
        v[2 * u + 1][nb] = make_float2(d[2], d[3]);
      }
    }
    // ---- digit 2 (chunk stride 1) and digit 3 (chunk stride 4) on slots
    if constexpr (G >= 64) {
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int a = 0; a < 16; a += 4) h4_stage(v[a][q], v[a + 1][q], v[a + 2][q], v[a + 3][q]);
    }
    if constexpr (G >= 256) {
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int b = 0; b < 4; ++b) h4_stage(v[b][q], v[b + 4][q], v[b + 8][q], v[b + 12][q]);
    }
    // ---- digit 4 (G = 1024): the four superblocks of a group sit in the
    // lanes with g ^ {0, 1, 2, 3} (lane ^ 4c). A 4-lane transpose first: slot
    // s with s & 3 = c comes from lane ^ 4c, so afterwards slot 4h + c holds
    // superblock j ^ c (j = g & 3) of the one chunk ((4h) ^ 4 (g >> 2)) | j.
    // The radix-4 stage depends only on the XOR of its two digits, so it runs
    // on those four slots as they are, and each result stays in its slot.
    if constexpr (G == 1024) {
#pragma unroll
      for (int c = 1; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float2& x = v[4 * h + c][q];
            x.x = __shfl_xor_sync(0xffffffffu, x.x, 4 * c);
            x.y = __shfl_xor_sync(0xffffffffu, x.y, 4 * c);
          }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int h = 0; h < 4; ++h) h4_stage(v[4 * h][q], v[4 * h + 1][q], v[4 * h + 2][q], v[4 * h + 3][q]);
    }

    // ---- row absmax (taken here, or read below in the given-max mode)
    if constexpr (RAG) {
      // the maxima of the two rows, each over the lines that lie in it
      float m = 0.0f, m2 = 0.0f;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float mh = 0.0f;
#pragma unroll
        for (int s = 4 * h; s < 4 * h + 4; ++s) {
          mh = fmax3(mh, fabsf(v[s][0].x), fabsf(v[s][0].y));
          mh = fmax3(mh, fabsf(v[s][1].x), fabsf(v[s][1].y));
        }
        const bool second = (in2 >> h) & 1u;
        m = fmaxf(m, second ? 0.0f : mh);
        m2 = fmaxf(m2, second ? mh : 0.0f);
      }
      const unsigned grp = __match_any_sync(0xffffffffu, my_row);
      const unsigned mx = __reduce_max_sync(grp, __float_as_uint(m));
      if (sb_valid && lane == __ffs(grp) - 1) atomicMax(&rowmax[my_row], mx);
      const unsigned grp2 = __match_any_sync(0xffffffffu, my_row2);
      const unsigned mx2 = __reduce_max_sync(grp2, __float_as_uint(m2));
      if (sb_valid && lane == __ffs(grp2) - 1) atomicMax(&rowmax[my_row2], mx2);
    } else if constexpr (MODE != kRqGivenMax) {
      float m = 0.0f;
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        m = fmax3(m, fabsf(v[s][0].x), fabsf(v[s][0].y));
        m = fmax3(m, fabsf(v[s][1].x), fabsf(v[s][1].y));
      }
      const unsigned grp = __match_any_sync(0xffffffffu, my_row);
      const unsigned mx = __reduce_max_sync(grp, __float_as_uint(m));
      if (sb_valid && lane == __ffs(grp) - 1) atomicMax(&rowmax[my_row], mx);
    }
    // the bulk store that last read this tile's staging buffer is done with it
    if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncthreads();
    // every warp has read stage st (and its tile index): refill it
    if (tid == 0) {
      if (exhausted) {
        fill(st, ntiles);
      } else {
        fill(st, dyn_base + pending);
        if (!exhausted) pending = atomicAdd(claims, 1u);
      }
      // NB = 2: the previous tile's codes are complete (the barrier above)
      if (NB == 2 && prev_tile >= 0) store_tile(prev_tile, (it - 1) & 1);
    }
    const uint32_t bsel = NB == 2 ? static_cast<uint32_t>(it & 1) * buf_bytes : 0u;

    // ---- quantize into the staging buffers (4-byte code words, 8-byte fp16
    // pieces; both conflict-free), then one bulk copy per output
    if (sb_valid && (WQ || WH)) {
      float amax_u;  // the row maximum of the unnormalized rotation
      if constexpr (MODE == kRqGivenMax) {
        const long long grow = tile * R + my_row;
        amax_u = grow < M ? amax[grow] / kNorm : 0.0f;
      } else {
        amax_u = __uint_as_float(rowmax[my_row]);
      }
      const float inv = amax_u > 0.0f ? static_cast<float>(QM) / amax_u : 0.0f;
      float inv_b = inv;  // RAG: the multiplier of the superblock's second row
      if constexpr (RAG) {
        const float amax_b = __uint_as_float(rowmax[my_row2]);
        inv_b = amax_b > 0.0f ? static_cast<float>(QM) / amax_b : 0.0f;
      }
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const float inv_s = RAG && ((in2 >> (s >> 2)) & 1u) ? inv_b : inv;
        const float2 inv2 = make_float2(inv_s, inv_s);
        const float2 t0 = f2_fma(v[s][0], inv2, mg2);  // positions 4t, 4t + 1
        const float2 t1 = f2_fma(v[s][1], inv2, mg2);  // positions 4t + 2, 4t + 3
        if constexpr (QM == 7) {
          if constexpr (WQ) {  // four two's-complement nibbles, the first in the low bits
            const uint32_t n = (__float_as_uint(t0.x) & 0xFu) | ((__float_as_uint(t0.y) & 0xFu) << 4) |
                               ((__float_as_uint(t1.x) & 0xFu) << 8) | ((__float_as_uint(t1.y) & 0xFu) << 12);
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(q_at(s) + bsel), "h"(static_cast<unsigned short>(n))
                         : "memory");
          }
          if constexpr (WH) {
            const float2 c0 = f2_sub(t0, mg2), c1 = f2_sub(t1, mg2);
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(h_at(s) + bsel),
                         "r"(e4m3x2(c0.x, c0.y) | (e4m3x2(c1.x, c1.y) << 16))
                         : "memory");
          }
          continue;
        }
        if constexpr (WQ) {
          const uint32_t b01 = __byte_perm(__float_as_uint(t0.x), __float_as_uint(t0.y), 0x0040);
          const uint32_t b23 = __byte_perm(__float_as_uint(t1.x), __float_as_uint(t1.y), 0x0040);
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(q_at(s) + bsel), "r"(__byte_perm(b01, b23, 0x5410))
                       : "memory");
        }
        if constexpr (WH) {
          const float2 c0 = f2_sub(t0, mg2), c1 = f2_sub(t1, mg2);
          const __half2 h0 = __floats2half2_rn(c0.x, c0.y), h1 = __floats2half2_rn(c1.x, c1.y);
          asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(h_at(s) + bsel),
                       "r"(*reinterpret_cast<const uint32_t*>(&h0)), "r"(*reinterpret_cast<const uint32_t*>(&h1))
                       : "memory");
        }
      }
    }
    if constexpr (MODE == kRqAbsmax) {
      for (int i = tid; i < R; i += blockDim.x)
        if (tile * R + i < M) amax[tile * R + i] = __uint_as_float(rowmax[i]) * kNorm;
      continue;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // staging writes -> the bulk copy
    if constexpr (NB == 1) {
      __syncthreads();
      if (tid == 0) store_tile(tile, 0);
    }
    for (int i = tid; i < R; i += blockDim.x)
      if (tile * R + i < M)
        S[tile * R + i] = (MODE == kRqGivenMax ? amax[tile * R + i] / kNorm : __uint_as_float(rowmax[i])) / s_div;
    prev_tile = tile;
    prev_it = it;
  }
  if constexpr (NB == 2 && MODE != kRqAbsmax) {
    // the last tile's codes: every warp has written and fenced them
    __syncthreads();
    if (tid == 0 && prev_tile >= 0) store_tile(prev_tile, prev_it & 1);
  }
  if (tid == 0) {
    // the last bulk stores complete before the CTA (and its shared memory) ends
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    // this CTA's claims are over; the last CTA of the launch resets the slot
    __threadfence();
    if (atomicAdd(&g_rq_sched[slot][1], 1u) == gridDim.x - 1) {
      g_rq_sched[slot][0] = 0u;
      g_rq_sched[slot][1] = 0u;
    }
  }
}

// Puts every launch slot of the tensor-core kernel's tile hand-out back to
// zero (after a kernel gave up a wait; a completed launch restores its own).
cudaError_t rq_sched_reset() {
  static const unsigned int zero[kRqSchedSlots][2] = {};
  return cudaMemcpyToSymbol(g_rq_sched, zero, sizeof(zero));
}

// ================================================================ host =====

static float scale_divisor(int transform, int G, int qm) {
  if (transform == CONVROT_T_REGULAR_H4) return static_cast<float>(qm) * static_cast<float>(1 << (ilog2_c(G) / 2));
  if (transform == CONVROT_T_RHT) return static_cast<float>(qm * std::sqrt(static_cast<double>(G)));
  return static_cast<float>(qm);
}


// Rows per tile: the smallest R for which R*K/EPT threads fill whole warps
// (or nearly), within the thread, TMA box and shared-memory limits.
static bool choose_rows(int K, int ept, bool phase_c, int* R_out, int* NT_out) {
  int bestR = -1, bestNT = 0;
  double best_eff = -1.0;
  for (int R = 1; R <= 64; ++R) {
    if ((static_cast<long long>(R) * K) % ept) continue;
    const int NT = static_cast<int>(static_cast<long long>(R) * K / ept);
    if (NT > 384) break;
    const long long bytes = static_cast<long long>(R) * K * (phase_c ? 8 : 4);
    if (bytes > 100 * 1024) break;
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

template <int T, int G, int QM, bool XQ>
static cudaError_t launch_lane_x(const __nv_bfloat16* X, long long M, int K, long long ldx, const int8_t* signs,
                               int8_t* Q, float* S, __half* Q16, cudaStream_t st, bool* launched) {
  *launched = false;
  const int lines = K / 64;
  if (K % 64 != 0 || lines > 384 || M > 0x7fffffffLL) return cudaSuccess;
  int R = 0, NT = 0;
  if (!choose_rows(K, 64, false, &R, &NT)) return cudaSuccess;
  // A TMA box spans at most 256 lines: wider rows (one row per tile) arrive
  // in equal parts, each starting on a 1 KB boundary of the stage so the
  // 128B swizzle is the same as for one copy.
  const int parts = (lines + 255) / 256;
  const int box_lines = lines / parts;
  if (parts > 1 && (R != 1 || lines % parts != 0 || box_lines % 8 != 0)) return cudaSuccess;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaSuccess;
  // X viewed as [M][K/64][64] bf16; one box is one tile of R rows (or a part
  // of the one row).
  CUtensorMap map;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(lines), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(ldx) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_lines), static_cast<cuuint32_t>(R)};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(X), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;
  const int threads = (NT + 31) / 32 * 32;
  // a 128-byte slot for every thread: R * K * 2 bytes of lines (NT slots),
  // then the zeroed slots of the padding threads
  const int stage_bytes = ((threads * 128 + 1023) / 1024) * 1024;
  // the quad transpose needs 256 bytes per thread (one fp32 line)
  using C = LaneCfg<T, G, XQ>;
  const int tbytes = C::QT ? threads * 256 : 0;
  const int smem = 1024 + 2 * stage_bytes + tbytes + ((3 * R + 1) & ~1) * 4 + 2 * 8 + 16 + C::NPOS * 128;
  auto kern = rq_lane_kernel<T, G, QM, XQ>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(reinterpret_cast<const void*>(kern), threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaSuccess;
  const long long tiles = (M + R - 1) / R;
  // the fewest CTAs that still take every tile in the same number of rounds:
  // no partial last round in which most of the GPU would sit idle
  const long long slots = std::min<long long>(tiles, static_cast<long long>(per_sm) * device_sm_count());
  const long long rounds = (tiles + slots - 1) / slots;
  const long long grid = (tiles + rounds - 1) / rounds;
  kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(map, M, K, R, NT, signs, Q, S, Q16,
                                                             scale_divisor(T, G, QM), stage_bytes, tbytes,
                                                             box_lines, kDefaultSpinLimit);
  *launched = true;
  return cudaGetLastError();
}

// Tiles of the tensor-core kernel: R rows whose superblocks fill whole warps
// (or nearly), at least min_warps warps where the shape allows, at most
// kMmaMaxWarps warps and 48 KB per tile.
static bool choose_rows_mma(int K, int min_warps, int* R_out, int* nsb_out) {
  // R is a multiple of r0, so that a tile is a whole number of superblocks
  // (4 lines of 64): 1 when K is a multiple of 256, else 2 or 4
  const int lines = K / 64;
  const int r0 = lines % 4 == 0 ? 1 : lines % 2 == 0 ? 2 : 4;
  int bestR = -1;
  double best = -1.0;
  for (int R = r0; R <= 64; R += r0) {
    const int nsb = R * lines / 4;
    const int warps = (nsb + 7) / 8;
    if (warps > kMmaMaxWarps || static_cast<long long>(R) * K * 2 > 48 * 1024) break;
    const double eff = static_cast<double>(nsb) / (8.0 * warps);
    if (warps >= min_warps && eff >= 0.999) {
      bestR = R;
      break;
    }
    if (eff > best + 1e-9) {
      best = eff;
      bestR = R;
    }
  }
  if (bestR < 0) return false;
  *R_out = bestR;
  *nsb_out = bestR * lines / 4;
  return true;
}

template <int G, int STAGES, bool WQ, bool WH, int MODE, int QM, int NB, bool RAG>
static cudaError_t launch_mma_s(const CUtensorMap& map, long long M, int K, int R, int nsb, int box_lines, int8_t* Q,
                                float* S, __half* Q16, float* amax, cudaStream_t st, bool* launched) {
  const int threads = 32 * ((nsb + 7) / 8);
  const int stage_bytes = (R * K * 2 + 1023) / 1024 * 1024;
  const int out_bytes = QM == 127 ? (WQ ? R * K : 0) + (WH ? 2 * R * K : 0) : (WQ ? R * K / 2 : 0) + (WH ? R * K : 0);
  const int buf_bytes = (out_bytes + 1023) / 1024 * 1024;
  const int smem = 1024 + STAGES * stage_bytes + NB * buf_bytes + ((3 * R + 1) & ~1) * 4 + STAGES * 16;
  auto kern = rq_mma_kernel<G, STAGES, WQ, WH, MODE, QM, NB, RAG>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(reinterpret_cast<const void*>(kern), threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaSuccess;
  const long long tiles = (M + R - 1) / R;
  const long long slots = std::min<long long>(tiles, static_cast<long long>(per_sm) * device_sm_count());
  const long long rounds = (tiles + slots - 1) / slots;
  const long long grid = (tiles + rounds - 1) / rounds;
  static std::atomic<unsigned int> launches{0};
  const int slot = static_cast<int>(launches.fetch_add(1u, std::memory_order_relaxed) % kRqSchedSlots);
  kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(map, M, K, R, nsb, Q, S, Q16, amax,
                                                           scale_divisor(CONVROT_T_REGULAR_H4, G, QM), stage_bytes,
                                                           box_lines, slot, kDefaultSpinLimit);
  *launched = true;
  return cudaGetLastError();
}

// X viewed as [M][K / 64][64] bf16 with a box of R rows of box_lines lines
// (128B swizzle); false if the encoder is missing or refuses.
static bool make_x_map(const __nv_bfloat16* X, long long M, int K, long long ldx, int R, int box_lines,
                       CUtensorMap* map) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(K / 64), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(ldx) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_lines), static_cast<cuuint32_t>(R)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(X), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core kernel: regular Hadamard, int8 codes (and fp16 copy), K a
// multiple of 256 (1024 for G = 1024); for G <= 64 with codes and scales,
// also K a multiple of 64 from 256 up (a superblock then spans at most two
// rows of a tile). *launched stays false for shapes it does not take.
template <int G, int MODE, int QM>
static cudaError_t launch_mma(const __nv_bfloat16* X, long long M, int K, long long ldx, int8_t* Q, float* S,
                              __half* Q16, float* amax, cudaStream_t st, bool* launched) {
  *launched = false;
  if ((G == 1024 && K % 1024 != 0) || M > 0x7fffffffLL) return cudaSuccess;
  const bool rag = K % 256 != 0;
  if (rag && !(G <= 64 && MODE == kRqFull && K % 64 == 0 && K >= 256)) return cudaSuccess;
  // Tile shape by what the launch writes (GB300, one GPU, the DiT, qkv and
  // group-sweep activations). With the fp16 copy (or the e4m3 one) the
  // staging is large: 6-warp tiles of about 24 KB with 3 stages, 2 CTAs per
  // SM. With the codes alone (two small staging buffers) or nothing but the
  // row maxima: 3-warp tiles of about 12 KB with 2 stages, 4-5 CTAs per SM,
  // which took the qkv activation from 47.4 to 45.4 us.
  const bool light = MODE == kRqAbsmax || (Q && !Q16);
  int R = 0, nsb = 0;
  if (!choose_rows_mma(K, light ? 3 : kMmaMinWarps, &R, &nsb)) return cudaSuccess;
  const int lines = K / 64;
  const int parts = (lines + 255) / 256;
  const int box_lines = lines / parts;
  if (parts > 1 && (R != 1 || lines % parts != 0 || box_lines % 8 != 0)) return cudaSuccess;
  CUtensorMap map;
  if (!make_x_map(X, M, K, ldx, R, box_lines, &map)) return cudaSuccess;
  // stages: three (two tiles in flight behind the one being worked on) for
  // the large tiles, within about 72 KB of input staging per CTA; two for the
  // light launches, whose CTAs are smaller and more per SM. Two output
  // staging buffers when the codes alone are written (the fp16 copy's would
  // cost a CTA per SM).
  const bool three = !light && R * K * 2 <= 24 * 1024;
#define CONVROT_RQ_MMA_R(WQ, WH, RG)                                                                               \
  return three ? launch_mma_s<G, 3, WQ, WH, MODE, QM, (WQ && !WH) ? 2 : 1, RG>(map, M, K, R, nsb, box_lines, Q, S,   \
                                                                               Q16, amax, st, launched)             \
               : launch_mma_s<G, 2, WQ, WH, MODE, QM, (WQ && !WH) ? 2 : 1, RG>(map, M, K, R, nsb, box_lines, Q, S,   \
                                                                               Q16, amax, st, launched)
#define CONVROT_RQ_MMA(WQ, WH)                      \
  {                                                 \
    if constexpr (G <= 64 && MODE == kRqFull) {     \
      if (rag) CONVROT_RQ_MMA_R(WQ, WH, true);      \
    }                                               \
    CONVROT_RQ_MMA_R(WQ, WH, false);                \
  }
  if constexpr (MODE == kRqAbsmax) {
    CONVROT_RQ_MMA(false, false)
  } else {
    if (Q && Q16) CONVROT_RQ_MMA(true, true)
    if (Q16) CONVROT_RQ_MMA(false, true)
    CONVROT_RQ_MMA(true, false)
  }
#undef CONVROT_RQ_MMA
#undef CONVROT_RQ_MMA_R
}

template <int MODE, int QM = 127>
static cudaError_t launch_mma_any(const __nv_bfloat16* X, long long M, int K, long long ldx, int G, int8_t* Q,
                                  float* S, __half* Q16, float* amax, cudaStream_t st, bool* launched) {
  *launched = false;
  switch (G) {
    case 4: return launch_mma<4, MODE, QM>(X, M, K, ldx, Q, S, Q16, amax, st, launched);
    case 16: return launch_mma<16, MODE, QM>(X, M, K, ldx, Q, S, Q16, amax, st, launched);
    case 64: return launch_mma<64, MODE, QM>(X, M, K, ldx, Q, S, Q16, amax, st, launched);
    case 256: return launch_mma<256, MODE, QM>(X, M, K, ldx, Q, S, Q16, amax, st, launched);
    case 1024: return launch_mma<1024, MODE, QM>(X, M, K, ldx, Q, S, Q16, amax, st, launched);
    default: return cudaSuccess;
  }
}

// The randomized Hadamard's strides 64 and 128 go through the quad
// transpose when a row is a whole number of quads (K a multiple of 256): the
// stores then fill whole lines, as on the regular Hadamard path.
template <int T, int G, int QM>
static cudaError_t launch_lane(const __nv_bfloat16* X, long long M, int K, long long ldx, const int8_t* signs,
                               int8_t* Q, float* S, __half* Q16, cudaStream_t st, bool* launched) {
  if constexpr (T == CONVROT_T_RHT && G >= 128) {
    if (K % 256 == 0) return launch_lane_x<T, G, QM, true>(X, M, K, ldx, signs, Q, S, Q16, st, launched);
  }
  return launch_lane_x<T, G, QM, false>(X, M, K, ldx, signs, Q, S, Q16, st, launched);
}

// Entry used by the ABI layer. Returns a cudaError_t; *path tells which
// kernel ran (0 = generic, 1 = fast).
template <int QM>
static cudaError_t launch_lane_any(const __nv_bfloat16* xb, long long M, int K, long long ldx, int G, int transform,
                                  const int8_t* signs, int8_t* Q, float* S, __half* q16, cudaStream_t st,
                                  bool* launched) {
  constexpr int H4 = CONVROT_T_REGULAR_H4, RHT = CONVROT_T_RHT;
  *launched = false;
  if (transform == H4) {
    switch (G) {
      case 4: return launch_lane<H4, 4, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 16: return launch_lane<H4, 16, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 64: return launch_lane<H4, 64, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 256: return launch_lane<H4, 256, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 1024: return launch_lane<H4, 1024, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      default: return cudaSuccess;
    }
  }
  if (transform == RHT) {
    switch (G) {
      case 2: return launch_lane<RHT, 2, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 4: return launch_lane<RHT, 4, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 8: return launch_lane<RHT, 8, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 16: return launch_lane<RHT, 16, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 32: return launch_lane<RHT, 32, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 64: return launch_lane<RHT, 64, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 128: return launch_lane<RHT, 128, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      case 256: return launch_lane<RHT, 256, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
      default: return cudaSuccess;
    }
  }
  return launch_lane<CONVROT_T_NONE, 1, QM>(xb, M, K, ldx, signs, Q, S, q16, st, launched);
}

// qm = 127: int8 codes (Q) and fp16 copy (Q16), either but not both may be
// null; qm = 7: packed 4-bit codes (Q, K / 2 bytes per row) and e4m3 copy
// (Q16 as bytes). kernel: kRqAuto picks the fastest kernel that takes the
// shape; the others ask for one kernel (a diagnostic): *path = -1 if it does
// not take the shape, else 0 = generic, 1 = register butterfly, 2 =
// tensor-core stage.
cudaError_t rotquant_launch(const void* X, int in_dtype, long long M, int K, long long ldx, int G, int transform,
                            const int8_t* signs, int8_t* Q, float* S, uint16_t* Q16, int kernel, int qm,
                            cudaStream_t st, int* path) {
  *path = 0;
  if (M <= 0) return cudaSuccess;
  __half* q16 = reinterpret_cast<__half*>(Q16);
  // the fast kernels read X by TMA (16-byte aligned base, row stride a
  // multiple of 16 bytes) and store 32-byte pieces
  const bool aligned32 = (reinterpret_cast<uintptr_t>(X) % 16 == 0) && (ldx % 8 == 0) &&
                         (reinterpret_cast<uintptr_t>(Q) % 32 == 0) &&
                         (Q16 == nullptr || reinterpret_cast<uintptr_t>(Q16) % 32 == 0);
  const bool fast_ok = in_dtype == CONVROT_DTYPE_BF16 && aligned32 && K % 16 == 0;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(X);
  if (fast_ok && transform == CONVROT_T_REGULAR_H4 && (kernel == kRqAuto || kernel == kRqMma)) {
    bool launched = false;
    cudaError_t e = qm == 7 ? launch_mma_any<kRqFull, 7>(xb, M, K, ldx, G, Q, S, q16, nullptr, st, &launched)
                            : launch_mma_any<kRqFull, 127>(xb, M, K, ldx, G, Q, S, q16, nullptr, st, &launched);
    if (e != cudaSuccess) return e;
    if (launched) {
      *path = 2;
      return cudaSuccess;
    }
  }
  if (kernel == kRqMma) {
    *path = -1;
    return cudaSuccess;
  }
  if (fast_ok && (kernel == kRqAuto || kernel == kRqLane)) {
    bool launched = false;
    cudaError_t e = qm == 7 ? launch_lane_any<7>(xb, M, K, ldx, G, transform, signs, Q, S, q16, st, &launched)
                            : launch_lane_any<127>(xb, M, K, ldx, G, transform, signs, Q, S, q16, st, &launched);
    if (e != cudaSuccess) return e;
    if (launched) {
      *path = 1;
      return cudaSuccess;
    }
  }
  if (kernel == kRqLane) {
    *path = -1;
    return cudaSuccess;
  }
  const int threads = 256;
  const size_t smem = static_cast<size_t>(K) * sizeof(float);
  const long long grid = std::min<long long>(M, 64LL * device_sm_count());
  const float sdiv = scale_divisor(transform, G, qm);
  if (in_dtype == CONVROT_DTYPE_BF16) {
    auto kern = rq_generic_kernel<__nv_bfloat16>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(static_cast<const __nv_bfloat16*>(X), M, K, ldx,
                                                             transform, G, signs, Q, S, q16, sdiv, qm);
  } else {
    auto kern = rq_generic_kernel<float>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid), threads, smem, st>>>(static_cast<const float*>(X), M, K, ldx, transform, G,
                                                             signs, Q, S, q16, sdiv, qm);
  }
  return cudaGetLastError();
}

// Row-parallel building blocks (regular Hadamard on the tensor-core kernel):
// give_max = false writes the row maxima of the rotated slice into amax;
// give_max = true quantizes with the row maxima read from amax. *launched
// is false for shapes the kernel does not take.
cudaError_t rotquant_sharded_launch(const void* X, long long M, int K, long long ldx, int G, bool give_max,
                                    float* amax, int8_t* Q, float* S, uint16_t* Q16, cudaStream_t st,
                                    bool* launched) {
  *launched = false;
  if (M <= 0) return cudaSuccess;
  if (reinterpret_cast<uintptr_t>(X) % 16 != 0 || ldx % 8 != 0 || reinterpret_cast<uintptr_t>(Q) % 32 != 0 ||
      reinterpret_cast<uintptr_t>(Q16) % 32 != 0)
    return cudaSuccess;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(X);
  __half* q16 = reinterpret_cast<__half*>(Q16);
  if (give_max) return launch_mma_any<kRqGivenMax>(xb, M, K, ldx, G, Q, S, q16, amax, st, launched);
  return launch_mma_any<kRqAbsmax>(xb, M, K, ldx, G, nullptr, nullptr, nullptr, amax, st, launched);
}

}  // namespace convrot
