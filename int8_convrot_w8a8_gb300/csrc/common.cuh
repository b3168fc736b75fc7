// Internal helpers shared by the CUDA translation units of libconvrot.
// Nothing here is part of the public ABI (see include/convrot.h).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/convrot.h"

namespace convrot {

// ---------------------------------------------------------------- status ----
// Each translation unit owns a device error word (internal linkage, no
// relocatable device code needed). Kernels record the first failure with
// atomicCAS; the host reads and clears every unit's word through the
// functions declared below.
#define CONVROT_DEFINE_STATUS_WORD(NAME)                                         \
  static __device__ int g_status_word;                                           \
  __device__ __forceinline__ void record_status(int code) {                      \
    atomicCAS(&g_status_word, 0, code);                                          \
  }                                                                              \
  int NAME() {                                                                   \
    int v = 0, z = 0;                                                            \
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess)     \
      return CONVROT_ERR_CUDA;                                                   \
    if (v != 0 && cudaMemcpyToSymbol(g_status_word, &z, sizeof(int)) != cudaSuccess) \
      return CONVROT_ERR_CUDA;                                                   \
    return v;                                                                    \
  }

int status_word_rotquant();

// Rotate+quantize kernel choice (rotquant_launch): the fastest kernel that
// takes the shape, or one kernel by name.
constexpr int kRqAuto = 0, kRqGeneric = 1, kRqLane = 2, kRqMma = 3;

// Host-side launch helpers. They remember, per device, the kernel attributes
// already set and the occupancy / SM-count queries already answered, so a
// call costs no repeated driver round trips. No device memory is involved.
cudaError_t set_smem_limit(const void* kernel, int bytes);
cudaError_t blocks_per_sm(const void* kernel, int threads, int smem_bytes, int* out);
int device_sm_count();
// Clusters of `cluster` CTAs of this kernel that can be resident at once.
cudaError_t max_active_clusters(const void* kernel, int threads, int smem_bytes, int cluster, int* out);

// The driver's cuTensorMapEncodeTiled, looked up once per process through
// the runtime (no link-time dependency on libcuda); nullptr if unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
int status_word_gemm_mma();
int status_word_gemm_tc();
int status_word_hmatmul();
int status_word_gemm_small();

// Spin limit of every bounded device-side wait (iterations of a try_wait
// loop with nanosleep back-off); about a second on a GB300.
constexpr long long kDefaultSpinLimit = 1ll << 22;

// ------------------------------------------------------------- small math --
__host__ __device__ constexpr int ilog2_c(int v) { return v <= 1 ? 0 : 1 + ilog2_c(v >> 1); }
__host__ __device__ constexpr int ilog4_c(int v) { return v <= 1 ? 0 : 1 + ilog4_c(v >> 2); }

// Rounding of a pre-scaled code to int8 without a conversion instruction:
// t = fma(y, inv, 1.5 * 2^23) is the exact product y*inv rounded once to the
// nearest integer (ties to even, since 1.5*2^23 is even and the fp32 ulp on
// [2^23, 2^24) is 1), and the low byte of t's bits is that integer in two's
// complement, valid for |y*inv| < 2^22.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4B400000u;

__device__ __forceinline__ int code_from_magic(float t) {
  return static_cast<int>(__float_as_uint(t) - kRoundMagicBits);
}

// ------------------------------------------------------- packed fp32 math --
// add/sub/fma on two fp32 lanes at once (sm_100+ packed fp32 pipe). Each lane
// is an ordinary IEEE fp32 operation, bit-identical to the scalar one.
__device__ __forceinline__ unsigned long long f2_pack(float2 a) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)), "l"(f2_pack(c)));
  return f2_unpack(r);
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------ memory ops --
struct alignas(32) U32x8 { uint32_t w[8]; };

// 32-byte read-only load (sm_100+), no L1 allocation: streaming input.
__device__ __forceinline__ U32x8 ldg_nc_256(const void* p) {
  U32x8 r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]),
                 "=r"(r.w[4]), "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p));
  return r;
}
__device__ __forceinline__ void stg_128(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// 32-byte store (sm_100+).
__device__ __forceinline__ void stg_256(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// bf16 pair in one 32-bit word -> two fp32 (exact widening).
__device__ __forceinline__ float bf16lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------ mbarriers ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// 3-D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
// Bounded wait on an mbarrier phase. Returns false after `limit` failed
// polls (the caller records CONVROT_ERR_TIMEOUT and winds down).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase, long long limit) {
  for (long long i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, phase)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

}  // namespace convrot
