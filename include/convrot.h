/*
 * convrot.h -- C ABI of the GB300 (sm_103a) INT8 ConvRot W8A8 linear layer.
 *
 * The layer (stable-diffusion.cpp docs "INT8 Convrot Safetensors",
 * sections "How INT8 convrot works", "Weight quantization",
 * "Runtime activation quantization"):
 *
 *   X_rot   = X R            R = block-diagonal, one normalized Kronecker power
 *                            of H4 per contiguous group of G input features
 *   s_x[r]  = max_i |X_rot[r,i]| / 127
 *   Q_x     = clamp(round(X_rot / s_x), -127, 127)            (int8)
 *   A[r,o]  = sum_i Q_x[r,i] * Q_w[o,i]                       (int32, exact)
 *   Y[r,o]  = A[r,o] * s_x[r] * s_w[o] + b[o]                 (bf16 out)
 *
 * with Q_w, s_w produced the same way from W_rot = W R, one scale per output
 * row. The block randomized Hadamard variant (gemma.cpp issue "Add
 * experimental W8A8 MatMul with optional QuaRot-style rotation", section
 * "Rotation method": +-1 signs, Walsh-Hadamard, 1/sqrt(B)) and the naive
 * variant without rotation share the same quantizer and GEMM.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are caller-allocated device memory; the library
 *    allocates no device memory and keeps no data between calls. It holds
 *    only the device error word read by convrot_get_device_status() and, on
 *    the host, per-device kernel attributes it has already set.
 *  - Work is enqueued on the given stream and runs asynchronously. Argument
 *    errors are detected on the host and returned BEFORE anything is
 *    launched; CONVROT_ERR_CUDA reports a failed launch.
 *  - Row-major layouts; K (the input-feature dimension) is contiguous.
 *  - Rounding is round-half-to-even. A row whose absmax is 0 gets scale 0 and
 *    all-zero codes. NaN/Inf inputs are outside the contract.
 *  - There is no CPU fallback and no silent fallback to an unquantized path:
 *    an unsupported configuration is an error.
 */
#ifndef CONVROT_H_
#define CONVROT_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CONVROT_OK = 0,
  CONVROT_ERR_INVALID_ARG = 1,       /* null pointer, bad size, mismatched operands */
  CONVROT_ERR_UNSUPPORTED_GROUP = 2, /* G not a power of 4 (or 2 for RHT), G does not divide K, or G too large */
  CONVROT_ERR_ALIGNMENT = 3,         /* pointer or leading dimension not aligned as documented */
  CONVROT_ERR_CUDA = 4,              /* a CUDA runtime call or kernel launch failed */
  CONVROT_ERR_TIMEOUT = 5            /* a bounded device-side wait gave up (see convrot_get_device_status) */
} convrot_status;

typedef enum {
  /* Regular Hadamard: normalized Kronecker power of H4, G = 4^n
   * ("INT8 Convrot Safetensors", "How INT8 convrot works"). */
  CONVROT_T_REGULAR_H4 = 0,
  /* Block randomized Hadamard: v -> H_B (D v) / sqrt(B), B = group = 2^m,
   * D = diag(signs), H_B the Walsh-Hadamard matrix in natural order
   * (gemma.cpp issue, "Rotation method"). */
  CONVROT_T_RHT = 1,
  /* No rotation: naive W8A8 (gemma.cpp issue, "Executive summary"). */
  CONVROT_T_NONE = 2
} convrot_transform;

enum { CONVROT_DTYPE_F32 = 0, CONVROT_DTYPE_BF16 = 1 };

/* Largest supported K (int32 accumulators cannot overflow: 127*127*K < 2^31
 * for K <= 133143; the kernels further bound it by on-chip storage). */
#define CONVROT_MAX_K 32768
/* Largest supported group size. */
#define CONVROT_MAX_GROUP 4096

/* Packed activation ("Runtime activation quantization": the I8 rows and
 * their floating-point row scales, reused by every linear with the same
 * input and group size). All pointers are device pointers.
 *   q      int8  [M, K], row stride K; 16-byte aligned.
 *   scale  fp32  [M].
 *   q_f16  fp16  [M, K] copy of q (integer-valued, exact) used as the
 *          tensor-core operand; may be NULL, in which case the linear runs
 *          the int8 warp-MMA path. 16-byte aligned. */
typedef struct {
  const int8_t* q;
  const float* scale;
  const uint16_t* q_f16;
  int64_t M;
  int64_t K;
  int32_t group;
  int32_t transform;
} convrot_packed_act;

/* Packed weight ("Weight quantization"): the same layout for the rotated,
 * per-output-row-quantized weight. All pointers are device pointers.
 *   q      int8  [N, K]; scale fp32 [N]; q_f16 fp16 [N, K] or NULL. */
typedef struct {
  const int8_t* q;
  const float* scale;
  const uint16_t* q_f16;
  int64_t N;
  int64_t K;
  int32_t group;
  int32_t transform;
} convrot_packed_weight;

/* Offline weight preparation ("How INT8 convrot works": W_rot = W R;
 * "Weight quantization": s_w[o] = max|W_rot[o,:]|/127,
 * Q_w = clamp(round(W_rot / s_w), -127, 127)).
 *   W       device, [N, K] row-major, dtype CONVROT_DTYPE_F32 or _BF16.
 *   signs   device int8 [group] of +-1 for CONVROT_T_RHT, else ignored (may be NULL).
 *   Qw      device int8 [N, K] (out).   sw  device fp32 [N] (out).
 *   Qw_f16  device fp16 [N, K] (out) or NULL.
 * Errors: INVALID_ARG (null/sizes), UNSUPPORTED_GROUP, ALIGNMENT (any pointer
 * not 16-byte aligned), CUDA. */
convrot_status convrot_prepare_weights(const void* W, int32_t w_dtype, int64_t N, int64_t K,
                                       int32_t group, int32_t transform, const int8_t* signs,
                                       int8_t* Qw, float* sw, uint16_t* Qw_f16,
                                       cudaStream_t stream);

/* Runtime activation rotation + per-row dynamic quantization
 * ("Runtime activation quantization"), fused in one kernel.
 *   X       device bf16 [M, K], row stride ldx elements (ldx >= K).
 *   signs   device int8 [group] for CONVROT_T_RHT, else ignored.
 *   Qx      device int8 [M, K] (out), sx device fp32 [M] (out),
 *   Qx_f16  device fp16 [M, K] (out) or NULL.
 * X must be 16-byte aligned with ldx a multiple of 8. The fast kernels run
 * when X is 16-byte aligned and Qx, Qx_f16 32-byte aligned: for the regular
 * Hadamard with K a multiple of 256 (1024 for G = 1024), or with G <= 64 and
 * K a multiple of 64 from 256 to 12288 (6144 when K / 64 is odd), the
 * tensor-core kernel (see
 * convrot_quantize_act_kernel), else the register butterfly, else the
 * generic kernel.
 * The tensor-core kernel hands its tiles out through a small counter array
 * of the library (one pair of counters per launch slot, 256 slots per
 * device, zero when the library is loaded; each completed launch puts its
 * slot back to zero; convrot_get_device_status() clears them all after a
 * timeout). Launches take the slots in turn, so at most 256 rotate+quantize
 * launches may be in flight on one device at the same time. A launch recorded
 * into a CUDA graph keeps the slot it was given: replays of one graph must
 * not overlap each other in time.
 * M == 0 is a no-op. */
convrot_status convrot_quantize_act(const void* X, int64_t M, int64_t K, int64_t ldx,
                                    int32_t group, int32_t transform, const int8_t* signs,
                                    int8_t* Qx, float* sx, uint16_t* Qx_f16,
                                    cudaStream_t stream);

/* convrot_quantize_act with the kernel chosen by the caller (a diagnostic
 * and test entry point; the pages have no counterpart). kernel:
 *   CONVROT_RQ_AUTO         what convrot_quantize_act runs (the fastest one
 *                           that takes the shape);
 *   CONVROT_RQ_GENERIC      one CTA per row, every stage through shared
 *                           memory (any transform, alignment and K);
 *   CONVROT_RQ_BUTTERFLY    the register kernel: every radix stage on fp32
 *                           registers, bit-identical to the generic kernel;
 *   CONVROT_RQ_TENSOR_CORE  the regular Hadamard with its 16-point stage on
 *                           the tensor cores (mma.sync bf16 -> fp32 from the
 *                           staged tile) and the higher digits on fp32
 *                           registers: G in {4, 16, 64, 256, 1024}, K a
 *                           multiple of 256 (1024 for G = 1024); for G <= 64
 *                           also K a multiple of 64 from 256 up (tiles of 2
 *                           or 4 rows of at most 48 KB, so up to 12288 when
 *                           K / 64 is even, 6144 when odd). The tensor
 *                           core sums its 16 exact products in fp32 in its own
 *                           order, so codes can differ from the butterfly's
 *                           by one where the value lies within a few fp32
 *                           ulps of a rounding boundary.
 * The fast kernels want X 16-byte and Qx, Qx_f16 32-byte aligned. Arguments
 * and errors as convrot_quantize_act, plus INVALID_ARG when the chosen kernel
 * does not take the shape or alignment (nothing is launched then). */
#define CONVROT_RQ_AUTO 0
#define CONVROT_RQ_GENERIC 1
#define CONVROT_RQ_BUTTERFLY 2
#define CONVROT_RQ_TENSOR_CORE 3
convrot_status convrot_quantize_act_kernel(const void* X, int64_t M, int64_t K, int64_t ldx,
                                           int32_t group, int32_t transform, const int8_t* signs,
                                           int8_t* Qx, float* sx, uint16_t* Qx_f16, int32_t kernel,
                                           cudaStream_t stream);

/* ---- Row-parallel (K-sharded) linear --------------------------------------
 * The sglang digest ("风险与影响") notes that tensor parallelism with row-
 * parallel linears splits the rotated input dimension, and requires each
 * rank's slice (input_size_per_partition) to be a whole number of groups. A
 * rank then holds X[:, K_r] and Q_w[:, K_r]. The row scale of
 * "Runtime activation quantization" is a maximum over the WHOLE row, and
 * A = sum_i Q_x Q_w is a sum over all of K, so the linear needs two
 * exchanges: an all-reduce (max) of every row's maximum, and an all-reduce
 * (sum) of the int32 partial accumulators, which is exact. These three calls
 * are the per-rank steps around those exchanges; the exchanges themselves are
 * the caller's (NCCL, or any other all-reduce). With the slices of one row
 * and weights prepared on the whole K (then sliced by columns):
 *   1. convrot_rotate_absmax on X[:, K_r]            -> amax_r [M]
 *   2. all-reduce max over ranks                     -> amax   [M]
 *   3. convrot_quantize_act_given_max(X[:, K_r], amax) -> Q_x,r and s_x
 *   4. convrot_gemm_s32(Q_x,r, Q_w[:, K_r])          -> A_r int32 [M, N]
 *   5. all-reduce sum over ranks                     -> A
 *   6. convrot_dequant(A, s_x, s_w, b)               -> Y bf16
 * gives codes, scales, A and Y bit-identical to the one-device path on the
 * whole row (the row maximum and the int32 sums are exact, and every value
 * is computed from the same operations).
 * Regular Hadamard only (the tensor-core kernel): each slice's K a multiple
 * of 256 (1024 for G = 1024); X 16-byte aligned, ldx a multiple of 8, Qx and
 * Qx_f16 32-byte aligned. UNSUPPORTED_GROUP for other transforms or slice
 * widths.
 *
 * convrot_rotate_absmax: amax[r] = max_i |X_rot[r, i]| over the given columns
 *   (the normalized rotation), fp32 [M] on the device.
 * convrot_quantize_act_given_max: as convrot_quantize_act, with the row
 *   maxima read from amax (fp32 [M], normalized as above) instead of taken
 *   over the given columns: s_x = amax / 127, Q_x = round(X_rot / s_x).
 * convrot_dequant: Y[r, o] = bf16(fma(float(A[r, o]), s_x[r] * s_w[o], b[o]))
 *   for int32 A [M, N] (row stride lda, a multiple of 4, 16-byte aligned),
 *   the same expression and rounding as the GEMM epilogues. bias may be NULL;
 *   Y bf16 [M, N], ldy a multiple of 8, 16-byte aligned. */
convrot_status convrot_rotate_absmax(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                    int32_t transform, float* amax, cudaStream_t stream);
convrot_status convrot_quantize_act_given_max(const void* X, int64_t M, int64_t K, int64_t ldx,
                                              int32_t group, int32_t transform, const float* amax,
                                              int8_t* Qx, float* sx, uint16_t* Qx_f16,
                                              cudaStream_t stream);
convrot_status convrot_dequant(const int32_t* A, int64_t M, int64_t N, int64_t lda, const float* sx,
                               const float* sw, const float* bias, uint16_t* Y, int64_t ldy,
                               cudaStream_t stream);

/* The H-as-a-matrix variant of convrot_quantize_act: each group is multiplied
 * by the dense G x G rotation on the tensor cores ("feat: load ConvRot int4
 * and per-channel int8 safetensors", section "The rotation": the rotation
 * applied as one matmul against a shared constant), then quantized as above.
 * Same arguments and results (up to fp32 rounding) as convrot_quantize_act;
 * CONVROT_T_REGULAR_H4 with G in {16, 64, 256} only, X dense (ldx == K),
 * K / max(G, 64) <= 128, Qx and Qx_f16 32-byte aligned. Kept for comparison. */
convrot_status convrot_quantize_act_hmatmul(const void* X, int64_t M, int64_t K, int64_t ldx,
                                            int32_t group, int8_t* Qx, float* sx,
                                            uint16_t* Qx_f16, cudaStream_t stream);

/* One linear: Y = A * s_x * s_w + b in bf16 ("Runtime activation
 * quantization", reconstruction).
 *   a, w    host pointers to descriptors of device data; a->K == w->K and
 *           the group/transform of both must match.
 *   bias    device fp32 [N] or NULL, 16-byte aligned (as must be w->scale).
 *   Y       device bf16 [M, N], row stride ldy >= N (multiple of 8, 16-byte aligned).
 * Paths, chosen by M and K:
 *   M <= 64      streams the int8 weights: 17..64 rows with K a multiple of
 *                128 on the tcgen05 tensor cores (weights and codes widened
 *                to fp16 on chip), otherwise with warp-level int8 MMA;
 *   M > 64       the 2-SM tcgen05 tensor-core GEMM when K is a multiple of
 *                64. It reads the fp16 operand copies, so a->q_f16 and
 *                w->q_f16 are REQUIRED there: without them the call returns
 *                INVALID_ARG (it never drops silently to a slower kernel);
 *   M > 64, K not a multiple of 64: the int8 warp-MMA GEMM (~150 TOPS on
 *                GB300), the only path for such shapes.
 * convrot_linear_multi_int8mma / convrot_gemm_s32_int8mma run the int8
 * warp-MMA GEMM for any shape when asked for by name. */
convrot_status convrot_linear(const convrot_packed_act* a, const convrot_packed_weight* w,
                              const float* bias, uint16_t* Y, int64_t ldy, cudaStream_t stream);

/* Several linears sharing one packed activation (qkv, gated-FFN pair:
 * "Runtime activation quantization" on packed-tensor reuse; gemma.cpp
 * "Implementation" on the fused gated-FFN pair), in one launch.
 *   n       number of linears, 1..8.
 *   w       host array [n] of weight descriptors.
 *   bias    host array [n] of device fp32 pointers (entries may be NULL), or NULL.
 *   Y       host array [n] of device bf16 outputs; ldy host array [n]. */
convrot_status convrot_linear_multi(const convrot_packed_act* a, int32_t n,
                                    const convrot_packed_weight* w, const float* const* bias,
                                    uint16_t* const* Y, const int64_t* ldy,
                                    cudaStream_t stream);

/* Raw int32 accumulators A = Q_x Q_w^T through the same GEMM main loop the
 * linear uses (no scaling). A device int32 [M, N], row stride lda >= N.
 * Test and diagnostic entry point. */
convrot_status convrot_gemm_s32(const convrot_packed_act* a, const convrot_packed_weight* w,
                                int32_t* A, int64_t lda, cudaStream_t stream);

/* The int8 warp-level MMA GEMM (mma.sync m16n8k32 with native int32
 * accumulation, ~150 TOPS on GB300, about 11x below the tensor-core path),
 * for any M and K, run only when a caller asks for it by name: it needs no
 * fp16 operand copies (q_f16 may be NULL). Arguments, results (bit-identical
 * to the other paths) and errors as convrot_linear_multi and
 * convrot_gemm_s32. */
convrot_status convrot_linear_multi_int8mma(const convrot_packed_act* a, int32_t n,
                                            const convrot_packed_weight* w, const float* const* bias,
                                            uint16_t* const* Y, const int64_t* ldy,
                                            cudaStream_t stream);
convrot_status convrot_gemm_s32_int8mma(const convrot_packed_act* a, const convrot_packed_weight* w,
                                        int32_t* A, int64_t lda, cudaStream_t stream);

/* GEMM workspace. The pages have no counterpart: this is a scheduling device
 * of the tensor-core path. When the tiles of the last round would leave at
 * least half of the GPU idle, the GEMM splits them along K, one piece per
 * cluster; the pieces add their int32 partial sums into the workspace and
 * the last one to arrive reads the totals and finishes the tile. Integer
 * sums are exact, so results are bit-identical with or without a workspace.
 *   workspace        device memory, 256-byte aligned, ALL ZERO before its
 *                    first use; every call whose kernels run to completion
 *                    leaves it all zero again (after a call that recorded
 *                    CONVROT_ERR_TIMEOUT its content is undefined: clear it).
 *   workspace_bytes  its size; CONVROT_GEMM_WORKSPACE_BYTES covers every split
 *                    the library plans on a GPU with up to 160 SMs, a smaller
 *                    one allows fewer. NULL: no split.
 * Calls sharing one workspace must not overlap in time (issue them on one
 * stream). The int8 warp-MMA and small-M paths ignore the workspace.
 * Errors as for the calls without _ws, plus ALIGNMENT (workspace) and
 * INVALID_ARG (negative size). */
#define CONVROT_GEMM_WORKSPACE_BYTES (4096 + 40 * 256 * 1024)

/* The schedule the large-M tensor-core GEMM uses for a shape, computed on the
 * host alone (no device call; a diagnostic and test entry point).
 *   M, K        rows and depth; bits 8 (the tensor-core path runs for M > 64
 *               and K a multiple of 64) or 4 (any M >= 1, K a multiple of 128).
 *   n, N        the n linears sharing the activation (host array of n widths).
 *   sms         SM count of the target GPU; one cluster is taken to be
 *               resident per SM pair (per SM when M <= 128, without pairs).
 *               The launch takes the resident count from the CUDA occupancy
 *               query instead, so this is the schedule a launch uses whenever
 *               that query returns sms / 2 (sms) clusters, as on a GB300
 *               with all 152 SMs free.
 *   workspace_bytes   the workspace size the call would be given (0: none).
 * Outputs: bn, the tile width (256, 224 or 192); whole_tiles, the tiles run
 * whole; split_tiles, the last round's tiles split along K (0: no split);
 * pieces, the K pieces of each split tile (1 without a split).
 * INVALID_ARG for a null pointer, n outside [1, 8], bits other than 8 or 4,
 * sms < 1, a negative workspace size, or a shape the path does not run
 * (including one with more tiles than one launch takes, 2^31 - 1). */
convrot_status convrot_gemm_tc_plan(int64_t M, int64_t K, int32_t n, const int64_t* N, int32_t bits,
                                    int32_t sms, int64_t workspace_bytes, int32_t* bn,
                                    int64_t* whole_tiles, int64_t* split_tiles, int32_t* pieces);

convrot_status convrot_linear_multi_ws(const convrot_packed_act* a, int32_t n,
                                       const convrot_packed_weight* w, const float* const* bias,
                                       uint16_t* const* Y, const int64_t* ldy, void* workspace,
                                       int64_t workspace_bytes, cudaStream_t stream);

convrot_status convrot_gemm_s32_ws(const convrot_packed_act* a, const convrot_packed_weight* w,
                                   int32_t* A, int64_t lda, void* workspace, int64_t workspace_bytes,
                                   cudaStream_t stream);

/* ---- The linear from the activation, in one call ---------------------------
 * The sglang digest's single fused op (its kitchen_int8.py excerpt: Hadamard
 * rotation -> dynamic per-row activation quantization -> INT8 GEMM -> dequant
 * epilogue -> bias), for n linears that share the input ("Runtime activation
 * quantization": one packed activation feeds every linear with the same input
 * and group size). The rotate+quantize kernel writes the packed activation
 * into the caller's scratch; the GEMM follows as its programmatic dependent
 * launch on the same stream. Results are bit-identical to
 * convrot_quantize_act followed by convrot_linear_multi_ws.
 *
 * convrot_int8_linear_scratch_bytes: the scratch size for M rows of K: the
 * int8 codes [M, K], the fp32 row scales [M] and, when the tensor-core path
 * runs (M > 64, K a multiple of 64), the fp16 operand copy [M, K], each part
 * starting on a 256-byte boundary. -1 for M < 0 or K outside [1, CONVROT_MAX_K].
 * When that path runs and every weight has its fp16 copy, the GEMM reads only
 * the fp16 copy and the int8 codes are not written (their region is left as
 * it was).
 *
 * convrot_int8_linear:
 *   X, M, K, ldx, group, transform, signs   as for convrot_quantize_act.
 *   n, w, bias, Y, ldy                      as for convrot_linear_multi; every
 *                                           w[i] must carry the same K, group
 *                                           and transform.
 *   scratch         device memory, 256-byte aligned, at least
 *                   convrot_int8_linear_scratch_bytes(M, K) bytes; owned by
 *                   the caller and overwritten by the call (it holds the
 *                   packed activation until the GEMM has read it, so calls on
 *                   different streams need different scratch).
 *   workspace, workspace_bytes   the optional GEMM workspace, as for
 *                   convrot_linear_multi_ws.
 * Every argument is checked on the host before anything is launched: errors as
 * for convrot_quantize_act and convrot_linear_multi_ws, plus INVALID_ARG
 * (scratch null or too small) and ALIGNMENT (scratch). M == 0 is a no-op. */
int64_t convrot_int8_linear_scratch_bytes(int64_t M, int64_t K);

convrot_status convrot_int8_linear(const void* X, int64_t M, int64_t K, int64_t ldx, int32_t group,
                                   int32_t transform, const int8_t* signs, int32_t n,
                                   const convrot_packed_weight* w, const float* const* bias, uint16_t* const* Y,
                                   const int64_t* ldy, void* scratch, int64_t scratch_bytes, void* workspace,
                                   int64_t workspace_bytes, cudaStream_t stream);

/* convrot_linear_multi with the GEMM workspace held by the library instead of
 * the caller: ALLOCATES NOTHING. The pages have no counterpart; this is a
 * deployment convenience of this library.
 * The scratch is a static device array of CONVROT_GEMM_WORKSPACE_BYTES, one
 * per device, zero when the library's module is loaded on that device. The
 * first call on each device locates it with cudaGetSymbolAddress (no device
 * work, no wait; make that first call before any stream capture, since it
 * may load the module). Every call whose kernels complete leaves it clear
 * again, and convrot_get_device_status() clears it whenever any kernel unit
 * recorded CONVROT_ERR_TIMEOUT. A split is planned only within that size (a
 * launch that would need more is rejected before it starts).
 * RACES: every caller on a device shares the one scratch. Calls that may
 * overlap in time on the GPU (different streams, different host threads)
 * race on it and can produce wrong results: serialize them, e.g. on one
 * stream, or give concurrent calls their own workspaces through
 * convrot_linear_multi_ws.
 * Errors: as convrot_linear_multi, plus CUDA if the scratch cannot be
 * located. */
convrot_status convrot_linear_multi_static(const convrot_packed_act* a, int32_t n,
                                           const convrot_packed_weight* w, const float* const* bias,
                                           uint16_t* const* Y, const int64_t* ldy, cudaStream_t stream);

/* ---- 4-bit ConvRot (W4A4) -------------------------------------------------
 * "feat: load ConvRot int4 and per-channel int8 safetensors", section
 * "Solution": codes in [-7, 7], one fp32 scale per output channel, adjacent
 * pairs packed in a byte; the rotation is the same as for int8 ("The
 * rotation"). Readings where the page is silent: element 2j sits in the low
 * nibble of byte j, as a two's-complement nibble; activations are quantized
 * per row like the int8 ones with 7 in place of 127 (s = max|x_rot| / 7).
 * The tensor cores read e4m3 copies of the codes (every integer in [-7, 7]
 * is exact in e4m3) through tcgen05 kind::f8f6f4, at twice the fp16 rate;
 * the int32 accumulators stay exact. K must be a multiple of 128.
 *   q4    packed codes [rows, K / 2] bytes (storage format; the GEMM reads q_f8)
 *   scale fp32 [rows]
 *   q_f8  e4m3 copy [rows, K] bytes (required by the GEMM), 16-byte aligned */
typedef struct {
  const uint8_t* q4;
  const float* scale;
  const uint8_t* q_f8;
  int64_t M;
  int64_t K;
  int32_t group;
  int32_t transform;
} convrot_packed_act4;

typedef struct {
  const uint8_t* q4;
  const float* scale;
  const uint8_t* q_f8;
  int64_t N;
  int64_t K;
  int32_t group;
  int32_t transform;
} convrot_packed_weight4;

/* convrot_prepare_weights with 4-bit codes: Qw4 [N, K / 2] bytes, sw fp32
 * [N], Qw_f8 e4m3 [N, K] or NULL. Errors as convrot_prepare_weights, plus
 * ALIGNMENT when K is not a multiple of 128. */
convrot_status convrot_prepare_weights4(const void* W, int32_t w_dtype, int64_t N, int64_t K,
                                        int32_t group, int32_t transform, const int8_t* signs,
                                        uint8_t* Qw4, float* sw, uint8_t* Qw_f8, cudaStream_t stream);

/* convrot_quantize_act with 4-bit codes: Qx4 [M, K / 2] bytes, sx fp32 [M],
 * Qx_f8 e4m3 [M, K] or NULL. The fastest path wants X 16-byte and Qx4,
 * Qx_f8 32-byte aligned. */
convrot_status convrot_quantize_act4(const void* X, int64_t M, int64_t K, int64_t ldx,
                                     int32_t group, int32_t transform, const int8_t* signs,
                                     uint8_t* Qx4, float* sx, uint8_t* Qx_f8, cudaStream_t stream);

/* Y = A * s_x * s_w + b (bf16) for n = 1..8 linears sharing one 4-bit
 * packed activation, on the e4m3 tensor-core path (any M >= 0). Workspace as
 * for convrot_linear_multi_ws (may be NULL). */
convrot_status convrot_linear4_multi(const convrot_packed_act4* a, int32_t n,
                                     const convrot_packed_weight4* w, const float* const* bias,
                                     uint16_t* const* Y, const int64_t* ldy, void* workspace,
                                     int64_t workspace_bytes, cudaStream_t stream);

/* Raw int32 accumulators of the 4-bit GEMM (tests). A int32 [M, N], lda >= N,
 * a multiple of 4. */
convrot_status convrot_gemm4_s32(const convrot_packed_act4* a, const convrot_packed_weight4* w,
                                 int32_t* A, int64_t lda, void* workspace, int64_t workspace_bytes,
                                 cudaStream_t stream);

/* Reads and clears the device error words of the current device (one per
 * kernel unit; synchronizes the device first). Every word is read and cleared
 * before anything is reported. If any holds CONVROT_ERR_TIMEOUT, the static
 * scratch of convrot_linear_multi_static is cleared (an aborted split can
 * leave partial sums there) and CONVROT_ERR_TIMEOUT is returned; otherwise
 * the first nonzero status, or CONVROT_OK if no kernel reported a problem.
 * convrot_last_error() then says how many units recorded a status. */
convrot_status convrot_get_device_status(void);

/* Test hook for the bounded waits: launches one block that waits on an
 * mbarrier nothing ever arrives on, with the given spin limit, on `stream`.
 * The wait gives up, records CONVROT_ERR_TIMEOUT in the device error word
 * and the kernel returns normally. */
convrot_status convrot_selftest_wait_timeout(int64_t spin_limit, cudaStream_t stream);

/* Static description of a status code. Never NULL. */
const char* convrot_status_str(convrot_status s);

/* Human-readable detail of the last error returned on this host thread. */
const char* convrot_last_error(void);

/* Library ABI version (major * 100 + minor). */
int32_t convrot_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONVROT_H_ */
