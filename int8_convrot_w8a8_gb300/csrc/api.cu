// extern "C" entry points of libconvrot: argument validation, path choice and
// launches. Every check happens on the host before anything is enqueued.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "gemm_common.cuh"

namespace convrot {

cudaError_t rotquant_launch(const void* X, int in_dtype, long long M, int K, long long ldx, int G, int transform,
                            const int8_t* signs, int8_t* Q, float* S, uint16_t* Q16, int kernel, int qm,
                            cudaStream_t st, int* path);
cudaError_t hmatmul_launch(const void* X, long long M, int K, long long ldx, int G, int8_t* Q, float* S,
                           uint16_t* Q16, cudaStream_t st);
bool hmatmul_supported(long long K, long long ldx, int G);
cudaError_t gemm_mma_launch(const int8_t* Qx, const float* sx, long long M, int K, const GemmOutputs& outs,
                            bool raw, cudaStream_t st);
cudaError_t gemm_tc_launch(const void* Qx16, const float* sx, long long M, int K, const GemmOutputs& outs, bool raw,
                           bool f8, void* ws, long long ws_bytes, cudaStream_t st);
bool gemm_tc_supported(long long M, int K);
bool gemm_tc_plan(long long M, int K, const GemmOutputs& outs, bool f8, int sms, long long ws_bytes, int* bn,
                  long long* whole, long long* split, int* pieces);
cudaError_t gemm_small_launch(const int8_t* Qx, const float* sx, long long M, int K, const GemmOutputs& outs,
                              bool raw, cudaStream_t st);
bool gemm_small_supported(long long M, int K);
cudaError_t gemm_small_tc_launch(const int8_t* Qx, const float* sx, long long M, int K, const GemmOutputs& outs,
                                 bool raw, cudaStream_t st);
bool gemm_small_tc_supported(long long M, int K);
int status_word_gemm_small_tc();
cudaError_t selftest_wait_launch(long long spin_limit, cudaStream_t st);
cudaError_t rq_sched_reset();
cudaError_t rotquant_sharded_launch(const void* X, long long M, int K, long long ldx, int G, bool give_max,
                                    float* amax, int8_t* Q, float* S, uint16_t* Q16, cudaStream_t st,
                                    bool* launched);
cudaError_t dequant_launch(const int32_t* A, long long M, int N, long long lda, const float* sx, const float* sw,
                           const float* bias, uint16_t* Y, long long ldy, cudaStream_t st);

CONVROT_DEFINE_STATUS_WORD(status_word_api)

// Scratch of convrot_linear_multi_static: the GEMM workspace as a static
// device array (one copy per device, zero when the module loads), so that
// entry point allocates nothing.
static __device__ __align__(256) unsigned char g_static_gemm_scratch[CONVROT_GEMM_WORKSPACE_BYTES];

namespace {
std::mutex g_cache_mu;
std::map<std::pair<const void*, int>, int> g_smem_set;                 // (kernel, device) -> bytes
std::map<std::tuple<const void*, int, int, int>, int> g_occupancy;     // (kernel, device, threads, smem)
std::map<int, int> g_sms;                                              // device -> SM count
std::map<std::tuple<const void*, int, int, int>, int> g_clusters;      // (kernel, device, smem, cluster)
std::map<int, void*> g_static_scratch;                                 // device -> scratch address
}  // namespace

cudaError_t set_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto it = g_smem_set.find({kernel, dev});
  if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_set[{kernel, dev}] = bytes;
  return e;
}

cudaError_t blocks_per_sm(const void* kernel, int threads, int smem_bytes, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto key = std::make_tuple(kernel, dev, threads, smem_bytes);
  auto it = g_occupancy.find(key);
  if (it != g_occupancy.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kernel, threads, smem_bytes);
  if (e == cudaSuccess) g_occupancy[key] = *out;
  return e;
}

cudaError_t max_active_clusters(const void* kernel, int threads, int smem_bytes, int cluster, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto key = std::make_tuple(kernel, dev, smem_bytes, cluster * 4096 + threads);
  auto it = g_clusters.find(key);
  if (it != g_clusters.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
  if (e == cudaSuccess) g_clusters[key] = *out;
  return e;
}

EncodeTiledFn tensor_map_encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n < 1) n = 1;
  g_sms[dev] = n;
  return n;
}

}  // namespace convrot

using namespace convrot;

namespace {

thread_local char g_last_error[512] = "";

convrot_status fail(convrot_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

convrot_status ok() {
  g_last_error[0] = '\0';
  return CONVROT_OK;
}

convrot_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CONVROT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, unsigned n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }
bool is_pow4(long long v) { return is_pow2(v) && (__builtin_ctzll(static_cast<unsigned long long>(v)) % 2) == 0; }

// Group rules: "INT8 Convrot Safetensors", "Checkpoint format" (power of
// four dividing the input features); gemma.cpp issue, "Rotation method"
// (block transform only when K is divisible by the block).
convrot_status check_shape(long long K, int group, int transform) {
  if (K <= 0 || K > CONVROT_MAX_K) return fail(CONVROT_ERR_INVALID_ARG, "K=%lld outside [1, %d]", K, CONVROT_MAX_K);
  if (K % 16) return fail(CONVROT_ERR_ALIGNMENT, "K=%lld must be a multiple of 16", K);
  switch (transform) {
    case CONVROT_T_REGULAR_H4:
      if (group < 4 || group > CONVROT_MAX_GROUP || !is_pow4(group))
        return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "group %d is not a power of four in [4, %d]", group,
                    CONVROT_MAX_GROUP);
      if (K % group) return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "group %d does not divide K=%lld", group, K);
      return CONVROT_OK;
    case CONVROT_T_RHT:
      if (group < 2 || group > CONVROT_MAX_GROUP || !is_pow2(group))
        return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "block %d is not a power of two in [2, %d]", group,
                    CONVROT_MAX_GROUP);
      if (K % group) return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "block %d does not divide K=%lld", group, K);
      return CONVROT_OK;
    case CONVROT_T_NONE:
      return CONVROT_OK;
    default:
      return fail(CONVROT_ERR_INVALID_ARG, "unknown transform %d", transform);
  }
}

convrot_status check_pair(const convrot_packed_act* a, const convrot_packed_weight* w) {
  if (!a || !w) return fail(CONVROT_ERR_INVALID_ARG, "null descriptor");
  if (a->M > 0 && (!a->q || !a->scale)) return fail(CONVROT_ERR_INVALID_ARG, "activation q/scale is null");
  if (!w->q || !w->scale) return fail(CONVROT_ERR_INVALID_ARG, "weight q/scale is null");
  if (a->M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(a->M));
  if (w->N <= 0) return fail(CONVROT_ERR_INVALID_ARG, "N=%lld must be >= 1", static_cast<long long>(w->N));
  if (a->K != w->K)
    return fail(CONVROT_ERR_INVALID_ARG, "K mismatch: activation %lld, weight %lld", static_cast<long long>(a->K),
                static_cast<long long>(w->K));
  if (a->transform != w->transform || (a->transform != CONVROT_T_NONE && a->group != w->group))
    return fail(CONVROT_ERR_INVALID_ARG, "activation and weight were rotated differently (group %d/%d, transform %d/%d)",
                a->group, w->group, a->transform, w->transform);
  convrot_status s = check_shape(a->K, a->group, a->transform);
  if (s != CONVROT_OK) return s;
  if (!aligned(a->q, 16) || !aligned(w->q, 16) || (a->q_f16 && !aligned(a->q_f16, 16)) ||
      (w->q_f16 && !aligned(w->q_f16, 16)))
    return fail(CONVROT_ERR_ALIGNMENT, "operand pointers must be 16-byte aligned");
  if (!aligned(a->scale, 4) || !aligned(w->scale, 16))
    return fail(CONVROT_ERR_ALIGNMENT, "activation scales must be 4-byte and weight scales 16-byte aligned");
  return CONVROT_OK;
}

// Path choice. M <= 64 streams the int8 weights (tcgen05 for 17..64 rows
// with K a multiple of 128, warp MMA otherwise). Larger M runs the 2-SM
// tensor-core GEMM, which reads the fp16 operand copies: a call without them
// is an error rather than a silent detour through the int8 warp-MMA kernel,
// about 11x slower on GB300, which a caller gets only by asking for it
// (int8_mma) or for shapes the tensor-core path does not take (K not a
// multiple of 64), where it is the only path.
convrot_status run_gemm(const convrot_packed_act* a, GemmOutputs& outs, bool raw, void* ws, long long ws_bytes,
                        cudaStream_t stream, bool int8_mma = false) {
  if (a->M == 0) return ok();
  bool all_f16 = a->q_f16 != nullptr;
  for (int i = 0; i < outs.count; ++i) all_f16 = all_f16 && outs.o[i].qw16 != nullptr;
  const int K = static_cast<int>(a->K);
  cudaError_t e;
  if (int8_mma) {
    e = gemm_mma_launch(a->q, a->scale, a->M, K, outs, raw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "int8 MMA GEMM launch");
  } else if (gemm_small_tc_supported(a->M, K)) {
    // a handful of rows, K a multiple of 128: the int8 weight stream widened
    // to fp16 on chip for the tcgen05 tensor cores
    e = gemm_small_tc_launch(a->q, a->scale, a->M, K, outs, raw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "small-M tensor-core GEMM launch");
  } else if (gemm_small_supported(a->M, K)) {
    // a handful of rows: the int8 weight stream, no fp16 copies needed
    e = gemm_small_launch(a->q, a->scale, a->M, K, outs, raw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "small-M GEMM launch");
  } else if (gemm_tc_supported(a->M, K)) {
    if (!all_f16)
      return fail(CONVROT_ERR_INVALID_ARG,
                  "M=%lld runs the tensor-core GEMM, which reads the fp16 operand copies: give q_f16 for the "
                  "activation and every weight (the int8 warp-MMA path runs only when asked for by name)",
                  static_cast<long long>(a->M));
    e = gemm_tc_launch(a->q_f16, a->scale, a->M, K, outs, raw, false, ws, ws_bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core GEMM launch");
  } else {
    e = gemm_mma_launch(a->q, a->scale, a->M, K, outs, raw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "int8 MMA GEMM launch");
  }
  return ok();
}

}  // namespace

extern "C" {

int32_t convrot_version(void) { return 102; }

const char* convrot_status_str(convrot_status s) {
  switch (s) {
    case CONVROT_OK: return "ok";
    case CONVROT_ERR_INVALID_ARG: return "invalid argument";
    case CONVROT_ERR_UNSUPPORTED_GROUP: return "unsupported group size";
    case CONVROT_ERR_ALIGNMENT: return "misaligned pointer or size";
    case CONVROT_ERR_CUDA: return "CUDA error";
    case CONVROT_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* convrot_last_error(void) { return g_last_error; }

convrot_status convrot_prepare_weights(const void* W, int32_t w_dtype, int64_t N, int64_t K, int32_t group,
                                       int32_t transform, const int8_t* signs, int8_t* Qw, float* sw,
                                       uint16_t* Qw_f16, cudaStream_t stream) {
  if (!W || !Qw || !sw) return fail(CONVROT_ERR_INVALID_ARG, "W, Qw and sw must be non-null");
  if (w_dtype != CONVROT_DTYPE_F32 && w_dtype != CONVROT_DTYPE_BF16)
    return fail(CONVROT_ERR_INVALID_ARG, "w_dtype %d is neither fp32 nor bf16", w_dtype);
  if (N <= 0) return fail(CONVROT_ERR_INVALID_ARG, "N=%lld must be >= 1", static_cast<long long>(N));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (transform == CONVROT_T_RHT && !signs) return fail(CONVROT_ERR_INVALID_ARG, "RHT needs the sign vector");
  if (!aligned(W, 16) || !aligned(Qw, 16) || !aligned(sw, 4) || (Qw_f16 && !aligned(Qw_f16, 16)))
    return fail(CONVROT_ERR_ALIGNMENT, "pointers must be 16-byte aligned (scales 4-byte)");
  int path = 0;
  cudaError_t e = rotquant_launch(W, w_dtype, N, static_cast<int>(K), K, group, transform, signs, Qw, sw, Qw_f16,
                                  w_dtype == CONVROT_DTYPE_F32 ? kRqGeneric : kRqAuto, 127, stream, &path);
  if (e != cudaSuccess) return cuda_fail(e, "weight rotate/quantize launch");
  return ok();
}

convrot_status convrot_quantize_act(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                    int32_t transform, const int8_t* signs, int8_t* Qx, float* sx,
                                    uint16_t* Qx_f16, cudaStream_t stream) {
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (M == 0) return ok();
  if (!X || !Qx || !sx) return fail(CONVROT_ERR_INVALID_ARG, "X, Qx and sx must be non-null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (transform == CONVROT_T_RHT && !signs) return fail(CONVROT_ERR_INVALID_ARG, "RHT needs the sign vector");
  if (!aligned(X, 16) || ldx % 8 || !aligned(Qx, 16) || !aligned(sx, 4) || (Qx_f16 && !aligned(Qx_f16, 16)))
    return fail(CONVROT_ERR_ALIGNMENT, "X, Qx, Qx_f16 must be 16-byte aligned and ldx a multiple of 8");
  int path = 0;
  cudaError_t e = rotquant_launch(X, CONVROT_DTYPE_BF16, M, static_cast<int>(K), ldx, group, transform, signs, Qx,
                                  sx, Qx_f16, 0, 127, stream, &path);
  if (e != cudaSuccess) return cuda_fail(e, "activation rotate/quantize launch");
  return ok();
}

convrot_status convrot_quantize_act_kernel(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                           int32_t transform, const int8_t* signs, int8_t* Qx, float* sx,
                                           uint16_t* Qx_f16, int32_t kernel, cudaStream_t stream) {
  if (kernel < CONVROT_RQ_AUTO || kernel > CONVROT_RQ_TENSOR_CORE)
    return fail(CONVROT_ERR_INVALID_ARG, "kernel %d is not a rotate+quantize kernel choice", kernel);
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (M == 0) return ok();
  if (!X || !Qx || !sx) return fail(CONVROT_ERR_INVALID_ARG, "X, Qx and sx must be non-null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (transform == CONVROT_T_RHT && !signs) return fail(CONVROT_ERR_INVALID_ARG, "RHT needs the sign vector");
  if (!aligned(X, 16) || ldx % 8 || !aligned(Qx, 16) || !aligned(sx, 4) || (Qx_f16 && !aligned(Qx_f16, 16)))
    return fail(CONVROT_ERR_ALIGNMENT, "X, Qx, Qx_f16 must be 16-byte aligned and ldx a multiple of 8");
  static_assert(CONVROT_RQ_GENERIC == kRqGeneric && CONVROT_RQ_BUTTERFLY == kRqLane &&
                    CONVROT_RQ_TENSOR_CORE == kRqMma && CONVROT_RQ_AUTO == kRqAuto,
                "kernel choice constants");
  int path = 0;
  cudaError_t e = rotquant_launch(X, CONVROT_DTYPE_BF16, M, static_cast<int>(K), ldx, group, transform, signs, Qx,
                                  sx, Qx_f16, kernel, 127, stream, &path);
  if (e != cudaSuccess) return cuda_fail(e, "activation rotate/quantize launch");
  if (path < 0)
    return fail(CONVROT_ERR_INVALID_ARG, "kernel %d does not take this shape (transform %d, G=%d, K=%lld, alignment)",
                kernel, transform, group, static_cast<long long>(K));
  return ok();
}

convrot_status convrot_rotate_absmax(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                    int32_t transform, float* amax, cudaStream_t stream) {
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (transform != CONVROT_T_REGULAR_H4)
    return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "the row-parallel steps take the regular Hadamard only");
  if (M == 0) return ok();
  if (!X || !amax) return fail(CONVROT_ERR_INVALID_ARG, "X and amax must be non-null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (!aligned(X, 16) || ldx % 8 || !aligned(amax, 4))
    return fail(CONVROT_ERR_ALIGNMENT, "X must be 16-byte aligned, ldx a multiple of 8, amax 4-byte aligned");
  bool launched = false;
  cudaError_t e = rotquant_sharded_launch(X, M, static_cast<int>(K), ldx, group, false, amax, nullptr, nullptr,
                                          nullptr, stream, &launched);
  if (e != cudaSuccess) return cuda_fail(e, "row-max launch");
  if (!launched)
    return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "the row-parallel steps need K a multiple of 256 (1024 for G=1024)");
  return ok();
}

convrot_status convrot_quantize_act_given_max(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                              int32_t transform, const float* amax, int8_t* Qx, float* sx,
                                              uint16_t* Qx_f16, cudaStream_t stream) {
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (transform != CONVROT_T_REGULAR_H4)
    return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "the row-parallel steps take the regular Hadamard only");
  if (M == 0) return ok();
  if (!X || !amax || !Qx || !sx) return fail(CONVROT_ERR_INVALID_ARG, "X, amax, Qx and sx must be non-null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (!aligned(X, 16) || ldx % 8 || !aligned(amax, 4) || !aligned(Qx, 32) || !aligned(sx, 4) ||
      (Qx_f16 && !aligned(Qx_f16, 32)))
    return fail(CONVROT_ERR_ALIGNMENT, "X must be 16-byte aligned, Qx and Qx_f16 32-byte aligned, ldx a multiple of 8");
  bool launched = false;
  cudaError_t e = rotquant_sharded_launch(X, M, static_cast<int>(K), ldx, group, true, const_cast<float*>(amax), Qx,
                                          sx, Qx_f16, stream, &launched);
  if (e != cudaSuccess) return cuda_fail(e, "given-max rotate/quantize launch");
  if (!launched)
    return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "the row-parallel steps need K a multiple of 256 (1024 for G=1024)");
  return ok();
}

convrot_status convrot_dequant(const int32_t* A, int64_t M, int64_t N, int64_t lda, const float* sx,
                               const float* sw, const float* bias, uint16_t* Y, int64_t ldy, cudaStream_t stream) {
  if (M < 0 || N < 1 || N > 0x7fffffffLL)
    return fail(CONVROT_ERR_INVALID_ARG, "M=%lld, N=%lld", static_cast<long long>(M), static_cast<long long>(N));
  if (M == 0) return ok();
  if (!A || !sx || !sw || !Y) return fail(CONVROT_ERR_INVALID_ARG, "A, sx, sw and Y must be non-null");
  if (lda < N || ldy < N) return fail(CONVROT_ERR_INVALID_ARG, "lda and ldy must be >= N");
  if (!aligned(A, 16) || lda % 4 || !aligned(Y, 16) || ldy % 8 || !aligned(sx, 4) || !aligned(sw, 4) ||
      (bias && !aligned(bias, 4)))
    return fail(CONVROT_ERR_ALIGNMENT, "A and Y must be 16-byte aligned, lda a multiple of 4 and ldy of 8");
  cudaError_t e = dequant_launch(A, M, static_cast<int>(N), lda, sx, sw, bias, Y, ldy, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
  return ok();
}

convrot_status convrot_quantize_act_hmatmul(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                            int8_t* Qx, float* sx, uint16_t* Qx_f16, cudaStream_t stream) {
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, CONVROT_T_REGULAR_H4);
  if (s != CONVROT_OK) return s;
  if (group != 16 && group != 64 && group != 256)
    return fail(CONVROT_ERR_UNSUPPORTED_GROUP, "the matmul variant supports G in {16, 64, 256}, got %d", group);
  if (M == 0) return ok();
  if (!X || !Qx || !sx) return fail(CONVROT_ERR_INVALID_ARG, "X, Qx and sx must be non-null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (!aligned(X, 16) || ldx % 8 || !aligned(Qx, 32) || !aligned(sx, 4) || (Qx_f16 && !aligned(Qx_f16, 32)))
    return fail(CONVROT_ERR_ALIGNMENT, "X must be 16-byte aligned, Qx and Qx_f16 32-byte aligned, ldx a multiple of 8");
  if (!hmatmul_supported(K, ldx, group))
    return fail(CONVROT_ERR_INVALID_ARG, "the matmul variant needs dense X (ldx == K) and K / max(G, 64) <= 128");
  cudaError_t e = hmatmul_launch(X, M, static_cast<int>(K), ldx, group, Qx, sx, Qx_f16, stream);
  if (e != cudaSuccess) return cuda_fail(e, "matmul rotate/quantize launch");
  return ok();
}

}  // extern "C"

namespace {

// Locates this device's static scratch on first use (cudaGetSymbolAddress);
// later calls reuse the address. The array is zero when the module is
// loaded, which is the state the split GEMM expects, so nothing is cleared
// here and nothing waits on the device.
convrot_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto it = g_static_scratch.find(dev);
  if (it != g_static_scratch.end()) {
    *out = it->second;
    return ok();
  }
  void* p = nullptr;
  size_t bytes = 0;
  e = cudaGetSymbolAddress(&p, g_static_gemm_scratch);
  if (e == cudaSuccess) e = cudaGetSymbolSize(&bytes, g_static_gemm_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "locating the static GEMM scratch");
  if (bytes < static_cast<size_t>(CONVROT_GEMM_WORKSPACE_BYTES))
    return fail(CONVROT_ERR_INVALID_ARG, "static GEMM scratch is %zu bytes, below the workspace size", bytes);
  g_static_scratch[dev] = p;
  *out = p;
  return ok();
}

convrot_status check_workspace(const void* ws, int64_t ws_bytes) {
  if (!ws) return ok();
  if (!aligned(ws, 256)) return fail(CONVROT_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (ws_bytes < 0) return fail(CONVROT_ERR_INVALID_ARG, "workspace_bytes=%lld < 0", static_cast<long long>(ws_bytes));
  return ok();
}

// Checks n linears against the packed activation and fills the GEMM's
// output table; launches nothing.
convrot_status build_outputs(const convrot_packed_act* a, int32_t n, const convrot_packed_weight* w,
                             const float* const* bias, uint16_t* const* Y, const int64_t* ldy, void* ws,
                             int64_t ws_bytes, GemmOutputs* outs) {
  if (n < 1 || n > kMaxLinears) return fail(CONVROT_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, kMaxLinears);
  if (!w || !Y || !ldy) return fail(CONVROT_ERR_INVALID_ARG, "w, Y and ldy arrays must be non-null");
  convrot_status s = check_workspace(ws, ws_bytes);
  if (s != CONVROT_OK) return s;
  *outs = GemmOutputs{};
  outs->count = n;
  for (int i = 0; i < n; ++i) {
    s = check_pair(a, &w[i]);
    if (s != CONVROT_OK) return s;
    const float* b = bias ? bias[i] : nullptr;
    if (a->M > 0 && !Y[i]) return fail(CONVROT_ERR_INVALID_ARG, "Y[%d] is null", i);
    if (ldy[i] < w[i].N) return fail(CONVROT_ERR_INVALID_ARG, "ldy[%d] < N", i);
    if (!aligned(Y[i], 16) || ldy[i] % 8) return fail(CONVROT_ERR_ALIGNMENT, "Y[%d] alignment", i);
    if (b && !aligned(b, 16)) return fail(CONVROT_ERR_ALIGNMENT, "bias[%d] must be 16-byte aligned", i);
    outs->o[i] = GemmOut{w[i].q, w[i].q_f16, w[i].scale, b, Y[i], ldy[i], static_cast<int>(w[i].N), 0};
  }
  return CONVROT_OK;
}

convrot_status linear_multi(const convrot_packed_act* a, int32_t n, const convrot_packed_weight* w,
                            const float* const* bias, uint16_t* const* Y, const int64_t* ldy, void* ws,
                            int64_t ws_bytes, cudaStream_t stream, bool int8_mma = false) {
  GemmOutputs outs;
  convrot_status s = build_outputs(a, n, w, bias, Y, ldy, ws, ws_bytes, &outs);
  if (s != CONVROT_OK) return s;
  return run_gemm(a, outs, false, ws, ws_bytes, stream, int8_mma);
}

// The packed activation of convrot_int8_linear inside the caller's scratch:
// int8 codes [M, K], fp32 row scales [M], and the fp16 operand copy [M, K]
// when the tensor-core GEMM will read it; each part 256-byte aligned.
struct ActLayout {
  long long scale_off, f16_off, total;
  bool f16;
};
ActLayout act_layout(long long M, long long K) {
  auto up = [](long long v) { return (v + 255) / 256 * 256; };
  ActLayout l;
  l.scale_off = up(M * K);
  l.f16 = gemm_tc_supported(M, static_cast<int>(K));
  l.f16_off = l.scale_off + up(4 * M);
  l.total = l.f16_off + (l.f16 ? up(2 * M * K) : 0);
  return l;
}

// ---- 4-bit variant
convrot_status check_pair4(const convrot_packed_act4* a, const convrot_packed_weight4* w) {
  if (!a || !w) return fail(CONVROT_ERR_INVALID_ARG, "null descriptor");
  if (a->M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(a->M));
  if (w->N <= 0) return fail(CONVROT_ERR_INVALID_ARG, "N=%lld must be >= 1", static_cast<long long>(w->N));
  if ((a->M > 0 && (!a->q_f8 || !a->scale)) || !w->q_f8 || !w->scale)
    return fail(CONVROT_ERR_INVALID_ARG, "the 4-bit GEMM needs the e4m3 copies and the scales of both operands");
  if (a->K != w->K)
    return fail(CONVROT_ERR_INVALID_ARG, "K mismatch: activation %lld, weight %lld", static_cast<long long>(a->K),
                static_cast<long long>(w->K));
  if (a->transform != w->transform || (a->transform != CONVROT_T_NONE && a->group != w->group))
    return fail(CONVROT_ERR_INVALID_ARG, "activation and weight were rotated differently");
  convrot_status s = check_shape(a->K, a->group, a->transform);
  if (s != CONVROT_OK) return s;
  if (a->K % 128) return fail(CONVROT_ERR_ALIGNMENT, "the 4-bit path needs K a multiple of 128, got %lld",
                              static_cast<long long>(a->K));
  if ((a->M > 0 && !aligned(a->q_f8, 16)) || !aligned(w->q_f8, 16) || !aligned(w->scale, 16) ||
      (a->M > 0 && !aligned(a->scale, 4)))
    return fail(CONVROT_ERR_ALIGNMENT, "e4m3 copies and weight scales must be 16-byte aligned");
  return ok();
}

convrot_status gemm4(const convrot_packed_act4* a, int32_t n, const convrot_packed_weight4* w,
                     const float* const* bias, void* const* Y, const int64_t* ldy, bool raw, void* ws,
                     int64_t ws_bytes, cudaStream_t stream) {
  if (n < 1 || n > kMaxLinears) return fail(CONVROT_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, kMaxLinears);
  if (!w || !Y || !ldy) return fail(CONVROT_ERR_INVALID_ARG, "w, Y and ldy arrays must be non-null");
  convrot_status s = check_workspace(ws, ws_bytes);
  if (s != CONVROT_OK) return s;
  GemmOutputs outs{};
  outs.count = n;
  for (int i = 0; i < n; ++i) {
    s = check_pair4(a, &w[i]);
    if (s != CONVROT_OK) return s;
    const float* b = bias ? bias[i] : nullptr;
    if (a->M > 0 && !Y[i]) return fail(CONVROT_ERR_INVALID_ARG, "Y[%d] is null", i);
    if (ldy[i] < w[i].N) return fail(CONVROT_ERR_INVALID_ARG, "ldy[%d] < N", i);
    if (!aligned(Y[i], 16) || ldy[i] % (raw ? 4 : 8)) return fail(CONVROT_ERR_ALIGNMENT, "Y[%d] alignment", i);
    if (b && !aligned(b, 16)) return fail(CONVROT_ERR_ALIGNMENT, "bias[%d] must be 16-byte aligned", i);
    outs.o[i] = GemmOut{nullptr, reinterpret_cast<const uint16_t*>(w[i].q_f8), w[i].scale, b, Y[i], ldy[i],
                        static_cast<int>(w[i].N), 0};
  }
  if (a->M == 0) return ok();
  cudaError_t e = gemm_tc_launch(a->q_f8, a->scale, a->M, static_cast<int>(a->K), outs, raw, true, ws, ws_bytes,
                                 stream);
  if (e != cudaSuccess) return cuda_fail(e, "4-bit tensor-core GEMM launch");
  return ok();
}

convrot_status gemm_s32(const convrot_packed_act* a, const convrot_packed_weight* w, int32_t* A, int64_t lda,
                        void* ws, int64_t ws_bytes, cudaStream_t stream, bool int8_mma = false) {
  convrot_status s = check_pair(a, w);
  if (s != CONVROT_OK) return s;
  s = check_workspace(ws, ws_bytes);
  if (s != CONVROT_OK) return s;
  if (a->M > 0 && !A) return fail(CONVROT_ERR_INVALID_ARG, "A is null");
  if (lda < w->N) return fail(CONVROT_ERR_INVALID_ARG, "lda < N");
  if (!aligned(A, 16) || lda % 4) return fail(CONVROT_ERR_ALIGNMENT, "A must be 16-byte aligned and lda a multiple of 4");
  GemmOutputs outs{};
  outs.count = 1;
  outs.o[0] = GemmOut{w->q, w->q_f16, w->scale, nullptr, A, lda, static_cast<int>(w->N), 0};
  return run_gemm(a, outs, true, ws, ws_bytes, stream, int8_mma);
}

}  // namespace

extern "C" {

convrot_status convrot_linear(const convrot_packed_act* a, const convrot_packed_weight* w, const float* bias,
                              uint16_t* Y, int64_t ldy, cudaStream_t stream) {
  convrot_status s = check_pair(a, w);
  if (s != CONVROT_OK) return s;
  if (a->M > 0 && !Y) return fail(CONVROT_ERR_INVALID_ARG, "Y is null");
  if (ldy < w->N) return fail(CONVROT_ERR_INVALID_ARG, "ldy=%lld < N=%lld", static_cast<long long>(ldy), static_cast<long long>(w->N));
  if ((a->M > 0 && !aligned(Y, 16)) || ldy % 8) return fail(CONVROT_ERR_ALIGNMENT, "Y must be 16-byte aligned and ldy a multiple of 8");
  if (bias && !aligned(bias, 16)) return fail(CONVROT_ERR_ALIGNMENT, "bias must be 16-byte aligned");
  GemmOutputs outs{};
  outs.count = 1;
  outs.o[0] = GemmOut{w->q, w->q_f16, w->scale, bias, Y, ldy, static_cast<int>(w->N), 0};
  return run_gemm(a, outs, false, nullptr, 0, stream);
}

convrot_status convrot_linear_multi(const convrot_packed_act* a, int32_t n, const convrot_packed_weight* w,
                                    const float* const* bias, uint16_t* const* Y, const int64_t* ldy,
                                    cudaStream_t stream) {
  return linear_multi(a, n, w, bias, Y, ldy, nullptr, 0, stream);
}

convrot_status convrot_linear_multi_ws(const convrot_packed_act* a, int32_t n, const convrot_packed_weight* w,
                                       const float* const* bias, uint16_t* const* Y, const int64_t* ldy,
                                       void* workspace, int64_t workspace_bytes, cudaStream_t stream) {
  return linear_multi(a, n, w, bias, Y, ldy, workspace, workspace_bytes, stream);
}

int64_t convrot_int8_linear_scratch_bytes(int64_t M, int64_t K) {
  if (M < 0 || K <= 0 || K > CONVROT_MAX_K) return -1;
  return act_layout(M, K).total;
}

convrot_status convrot_int8_linear(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                   int32_t transform, const int8_t* signs, int32_t n,
                                   const convrot_packed_weight* w, const float* const* bias, uint16_t* const* Y,
                                   const int64_t* ldy, void* scratch, int64_t scratch_bytes, void* workspace,
                                   int64_t workspace_bytes, cudaStream_t stream) {
  // every argument is checked before the first launch
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (M > 0 && !X) return fail(CONVROT_ERR_INVALID_ARG, "X is null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (transform == CONVROT_T_RHT && !signs) return fail(CONVROT_ERR_INVALID_ARG, "RHT needs the sign vector");
  if (!aligned(X, 16) || ldx % 8) return fail(CONVROT_ERR_ALIGNMENT, "X must be 16-byte aligned and ldx a multiple of 8");
  const ActLayout l = act_layout(M, K);
  if (M > 0 && !scratch) return fail(CONVROT_ERR_INVALID_ARG, "scratch is null");
  if (!aligned(scratch, 256)) return fail(CONVROT_ERR_ALIGNMENT, "scratch must be 256-byte aligned");
  if (scratch_bytes < l.total)
    return fail(CONVROT_ERR_INVALID_ARG, "scratch_bytes=%lld < %lld needed", static_cast<long long>(scratch_bytes),
                l.total);
  char* base = static_cast<char*>(scratch);
  int8_t* q = reinterpret_cast<int8_t*>(base);
  float* sx = reinterpret_cast<float*>(base + l.scale_off);
  uint16_t* q16 = l.f16 ? reinterpret_cast<uint16_t*>(base + l.f16_off) : nullptr;
  const convrot_packed_act a{q, sx, q16, M, K, group, transform};
  GemmOutputs outs;
  s = build_outputs(&a, n, w, bias, Y, ldy, workspace, workspace_bytes, &outs);
  if (s != CONVROT_OK) return s;
  // the 2-SM tensor-core GEMM reads only the fp16 copies: every weight must
  // carry one (checked here, before the first launch); the int8 codes of the
  // activation are then not written
  const bool tc_only = q16 != nullptr;
  for (int i = 0; i < n && tc_only; ++i)
    if (!w[i].q_f16)
      return fail(CONVROT_ERR_INVALID_ARG,
                  "M=%lld runs the tensor-core GEMM, which reads the fp16 operand copies: weight %d has none",
                  static_cast<long long>(M), i);
  if (M == 0) return ok();
  int path = 0;
  cudaError_t e = rotquant_launch(X, CONVROT_DTYPE_BF16, M, static_cast<int>(K), ldx, group, transform, signs,
                                  tc_only ? nullptr : q, sx, q16, 0, 127, stream, &path);
  if (e != cudaSuccess) return cuda_fail(e, "activation rotate/quantize launch");
  // the GEMM is a programmatic dependent launch: its set-up and weight
  // prefetch overlap the rotate+quantize
  return run_gemm(&a, outs, false, workspace, workspace_bytes, stream);
}

convrot_status convrot_prepare_weights4(const void* W, int32_t w_dtype, int64_t N, int64_t K, int32_t group,
                                        int32_t transform, const int8_t* signs, uint8_t* Qw4, float* sw,
                                        uint8_t* Qw_f8, cudaStream_t stream) {
  if (!W || !Qw4 || !sw) return fail(CONVROT_ERR_INVALID_ARG, "W, Qw4 and sw must be non-null");
  if (w_dtype != CONVROT_DTYPE_F32 && w_dtype != CONVROT_DTYPE_BF16)
    return fail(CONVROT_ERR_INVALID_ARG, "w_dtype %d is neither fp32 nor bf16", w_dtype);
  if (N <= 0) return fail(CONVROT_ERR_INVALID_ARG, "N=%lld must be >= 1", static_cast<long long>(N));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (K % 128) return fail(CONVROT_ERR_ALIGNMENT, "the 4-bit path needs K a multiple of 128");
  if (transform == CONVROT_T_RHT && !signs) return fail(CONVROT_ERR_INVALID_ARG, "RHT needs the sign vector");
  if (!aligned(W, 16) || !aligned(Qw4, 16) || !aligned(sw, 4) || (Qw_f8 && !aligned(Qw_f8, 16)))
    return fail(CONVROT_ERR_ALIGNMENT, "pointers must be 16-byte aligned (scales 4-byte)");
  int path = 0;
  cudaError_t e = rotquant_launch(W, w_dtype, N, static_cast<int>(K), K, group, transform, signs,
                                  reinterpret_cast<int8_t*>(Qw4), sw, reinterpret_cast<uint16_t*>(Qw_f8),
                                  w_dtype == CONVROT_DTYPE_F32 ? kRqGeneric : kRqAuto, 7, stream, &path);
  if (e != cudaSuccess) return cuda_fail(e, "4-bit weight rotate/quantize launch");
  return ok();
}

convrot_status convrot_quantize_act4(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                     int32_t transform, const int8_t* signs, uint8_t* Qx4, float* sx, uint8_t* Qx_f8,
                                     cudaStream_t stream) {
  if (M < 0) return fail(CONVROT_ERR_INVALID_ARG, "M=%lld < 0", static_cast<long long>(M));
  convrot_status s = check_shape(K, group, transform);
  if (s != CONVROT_OK) return s;
  if (K % 128) return fail(CONVROT_ERR_ALIGNMENT, "the 4-bit path needs K a multiple of 128");
  if (M == 0) return ok();
  if (!X || !Qx4 || !sx) return fail(CONVROT_ERR_INVALID_ARG, "X, Qx4 and sx must be non-null");
  if (ldx < K) return fail(CONVROT_ERR_INVALID_ARG, "ldx=%lld < K=%lld", static_cast<long long>(ldx), static_cast<long long>(K));
  if (transform == CONVROT_T_RHT && !signs) return fail(CONVROT_ERR_INVALID_ARG, "RHT needs the sign vector");
  if (!aligned(X, 16) || ldx % 8 || !aligned(Qx4, 16) || !aligned(sx, 4) || (Qx_f8 && !aligned(Qx_f8, 16)))
    return fail(CONVROT_ERR_ALIGNMENT, "X, Qx4, Qx_f8 must be 16-byte aligned and ldx a multiple of 8");
  int path = 0;
  cudaError_t e = rotquant_launch(X, CONVROT_DTYPE_BF16, M, static_cast<int>(K), ldx, group, transform, signs,
                                  reinterpret_cast<int8_t*>(Qx4), sx, reinterpret_cast<uint16_t*>(Qx_f8), 0, 7, stream,
                                  &path);
  if (e != cudaSuccess) return cuda_fail(e, "4-bit activation rotate/quantize launch");
  return ok();
}

convrot_status convrot_linear4_multi(const convrot_packed_act4* a, int32_t n, const convrot_packed_weight4* w,
                                     const float* const* bias, uint16_t* const* Y, const int64_t* ldy,
                                     void* workspace, int64_t workspace_bytes, cudaStream_t stream) {
  return gemm4(a, n, w, bias, reinterpret_cast<void* const*>(Y), ldy, false, workspace, workspace_bytes, stream);
}

convrot_status convrot_gemm4_s32(const convrot_packed_act4* a, const convrot_packed_weight4* w, int32_t* A,
                                 int64_t lda, void* workspace, int64_t workspace_bytes, cudaStream_t stream) {
  void* y = A;
  return gemm4(a, 1, w, nullptr, &y, &lda, true, workspace, workspace_bytes, stream);
}

convrot_status convrot_linear_multi_static(const convrot_packed_act* a, int32_t n, const convrot_packed_weight* w,
                                           const float* const* bias, uint16_t* const* Y, const int64_t* ldy,
                                           cudaStream_t stream) {
  void* ws = nullptr;
  convrot_status s = static_scratch(&ws);
  if (s != CONVROT_OK) return s;
  return linear_multi(a, n, w, bias, Y, ldy, ws, CONVROT_GEMM_WORKSPACE_BYTES, stream);
}

convrot_status convrot_gemm_s32(const convrot_packed_act* a, const convrot_packed_weight* w, int32_t* A,
                                int64_t lda, cudaStream_t stream) {
  return gemm_s32(a, w, A, lda, nullptr, 0, stream);
}

convrot_status convrot_linear_multi_int8mma(const convrot_packed_act* a, int32_t n, const convrot_packed_weight* w,
                                            const float* const* bias, uint16_t* const* Y, const int64_t* ldy,
                                            cudaStream_t stream) {
  return linear_multi(a, n, w, bias, Y, ldy, nullptr, 0, stream, true);
}

convrot_status convrot_gemm_s32_int8mma(const convrot_packed_act* a, const convrot_packed_weight* w, int32_t* A,
                                        int64_t lda, cudaStream_t stream) {
  return gemm_s32(a, w, A, lda, nullptr, 0, stream, true);
}

convrot_status convrot_gemm_s32_ws(const convrot_packed_act* a, const convrot_packed_weight* w, int32_t* A,
                                   int64_t lda, void* workspace, int64_t workspace_bytes, cudaStream_t stream) {
  return gemm_s32(a, w, A, lda, workspace, workspace_bytes, stream);
}

convrot_status convrot_gemm_tc_plan(int64_t M, int64_t K, int32_t n, const int64_t* N, int32_t bits, int32_t sms,
                                    int64_t workspace_bytes, int32_t* bn, int64_t* whole_tiles, int64_t* split_tiles,
                                    int32_t* pieces) {
  if (!N || !bn || !whole_tiles || !split_tiles || !pieces) return fail(CONVROT_ERR_INVALID_ARG, "null argument");
  if (n < 1 || n > kMaxLinears) return fail(CONVROT_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, kMaxLinears);
  if (bits != 8 && bits != 4) return fail(CONVROT_ERR_INVALID_ARG, "bits=%d is neither 8 nor 4", bits);
  if (sms < 1) return fail(CONVROT_ERR_INVALID_ARG, "sms=%d < 1", sms);
  if (workspace_bytes < 0) return fail(CONVROT_ERR_INVALID_ARG, "negative workspace size");
  if (K < 1 || K > CONVROT_MAX_K) return fail(CONVROT_ERR_INVALID_ARG, "K=%lld outside [1, %d]",
                                               static_cast<long long>(K), CONVROT_MAX_K);
  if (bits == 8 ? !gemm_tc_supported(M, static_cast<int>(K)) : (M < 1 || K % 128 != 0))
    return fail(CONVROT_ERR_INVALID_ARG, "the tensor-core GEMM does not run for M=%lld, K=%lld at %d bits",
                static_cast<long long>(M), static_cast<long long>(K), bits);
  GemmOutputs outs{};
  outs.count = n;
  for (int i = 0; i < n; ++i) {
    if (N[i] < 1 || N[i] > 0x7fffffffLL) return fail(CONVROT_ERR_INVALID_ARG, "N[%d]=%lld", i, static_cast<long long>(N[i]));
    outs.o[i].n = static_cast<int>(N[i]);
  }
  int b = 0, pc = 0;
  long long wh = 0, sp = 0;
  if (!gemm_tc_plan(M, static_cast<int>(K), outs, bits == 4, sms, workspace_bytes, &b, &wh, &sp, &pc))
    return fail(CONVROT_ERR_INVALID_ARG, "no plan for this shape");
  *bn = b;
  *whole_tiles = wh;
  *split_tiles = sp;
  *pieces = pc;
  return ok();
}

convrot_status convrot_get_device_status(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  // every word is read (and so cleared) before anything is reported
  const int words[7] = {status_word_rotquant(), status_word_gemm_mma(),   status_word_gemm_tc(),
                        status_word_gemm_small(), status_word_gemm_small_tc(), status_word_hmatmul(),
                        status_word_api()};
  int first = 0, nonzero = 0;
  bool timeout = false;
  for (int w : words) {
    if (w == 0) continue;
    ++nonzero;
    if (first == 0) first = w;
    timeout = timeout || w == CONVROT_ERR_TIMEOUT;
  }
  if (timeout) {
    // an aborted split may have left partial sums and arrival counts in the
    // static scratch: clear it before any later call adds onto them
    int dev = 0;
    void* p = nullptr;
    if (cudaGetDevice(&dev) == cudaSuccess) {
      std::lock_guard<std::mutex> lock(g_cache_mu);
      auto it = g_static_scratch.find(dev);
      if (it != g_static_scratch.end()) p = it->second;
    }
    if (p) {
      e = cudaMemset(p, 0, CONVROT_GEMM_WORKSPACE_BYTES);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e, "clearing the static GEMM scratch");
    }
    // and the rotate+quantize tile hand-out counters
    e = rq_sched_reset();
    if (e != cudaSuccess) return cuda_fail(e, "clearing the tile hand-out counters");
  }
  if (first == 0) return ok();
  if (timeout && first != CONVROT_ERR_TIMEOUT) first = CONVROT_ERR_TIMEOUT;
  return fail(static_cast<convrot_status>(first), "%d kernel unit(s) recorded a status; reporting %d (%s)", nonzero,
              first, convrot_status_str(static_cast<convrot_status>(first)));
}

convrot_status convrot_selftest_wait_timeout(int64_t spin_limit, cudaStream_t stream) {
  if (spin_limit < 1 || spin_limit > (1ll << 30)) return fail(CONVROT_ERR_INVALID_ARG, "spin_limit out of range");
  cudaError_t e = selftest_wait_launch(spin_limit, stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ok();
}

}  // extern "C"

namespace convrot {

// One warp waits on an mbarrier that expects one arrival nobody makes. The
// bounded wait gives up, records CONVROT_ERR_TIMEOUT and the kernel ends.
__global__ void selftest_wait_kernel(long long spin_limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  __syncwarp();
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  const bool done = mbar_wait_bounded(&bar, 0, spin_limit);
  if (!done && threadIdx.x == 0) record_status(CONVROT_ERR_TIMEOUT);
}

cudaError_t selftest_wait_launch(long long spin_limit, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(spin_limit);
  return cudaGetLastError();
}

}  // namespace convrot
