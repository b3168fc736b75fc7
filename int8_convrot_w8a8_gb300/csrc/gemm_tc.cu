// Int8-exact GEMM on the 5th-generation tensor cores (tcgen05), with the
// dequant / bias / bf16 epilogue fused.
//
//   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]          (exact, int32)
//   Y[r, o] = bf16( fma(float(A[r,o]), s_x[r] * s_w[o], b[o]) )
//
// ("INT8 Convrot Safetensors", "Runtime activation quantization".)
//
// sm_103a has no integer tcgen05 MMA, so the int8 codes enter the tensor
// cores as fp16 values (every integer in [-127, 127] is exact in fp16) with
// an fp32 accumulator in tensor memory. Products are exact (|q*q| <= 16129)
// and so is every partial sum while it stays below 2^24 in magnitude:
// 127 * 127 * 1024 = 16 516 096 < 2^24 = 16 777 216. The K loop therefore
// runs in chunks of 16 stage rows (1024 fp16 K values); each chunk
// accumulates into a fresh TMEM buffer, and the epilogue warps convert the
// chunk (an exact integer in fp32) to int32 and add it into int32 registers.
// Two TMEM buffers alternate, so the tensor cores fill chunk c+1 while chunk
// c drains. The 4-bit codes of the W4A4 variant ("feat: load ConvRot int4
// and per-channel int8 safetensors", "Solution": values in [-7, 7]) enter as
// e4m3 (exact) through kind::f8f6f4 at twice the fp16 rate; a 128-byte stage
// row then holds 128 K values, and |q*q| <= 49 keeps every partial sum of any
// supported K exact, so a tile accumulates in one chunk.
//
// Structure (one persistent CTA per SM, 320 threads; CTA pairs when M > 128):
//   warp 0      TMA producer: 128 A rows and BN / CL B rows per stage (128
//               bytes of K each, 128-byte swizzle) into a STAGES-deep ring;
//               in a pair both CTAs' copies complete on the leader's barrier.
//   warp 1      TMEM allocation and the MMA issuer: tcgen05.mma, M = 128 * CL,
//               N = BN, four MMAs per stage row, cta_group::CL; in a pair only
//               the leader issues, and its commits are multicast to both.
//   warps 2..9  epilogue: TMEM -> registers (tcgen05.ld 32x32b), int32
//               accumulation; column scales and biases copied to shared
//               memory (cp.async) while the MMAs run; then scaling, bias,
//               bf16, and 32 x 16 TMA tiled stores of Y.
// Tiles are handed out statically (tile = blockIdx.x + i * gridDim.x) in a
// grouped order for L2 reuse. When the last round would leave most of the
// GPU idle and the caller gave a workspace, the tiles of that round are
// split along K instead, one piece per cluster, computed before the
// cluster's whole tiles: each piece adds its int32 partial sums into the
// tile's workspace slot with bulk reductions (TMA, performed in L2), and the
// warp that brings the last piece of its 32-row slab reads the totals back,
// clears them and runs the epilogue, all while the tensor cores move on to
// the whole tiles. Integer
// addition is exact and associative, so the result is bit-identical to the
// unsplit schedule and does not depend on how the rows are partitioned.
// Nothing waits on another CTA.
//
// Every mbarrier wait is bounded. A wait that gives up records
// CONVROT_ERR_TIMEOUT in the device error word and raises a CTA-wide abort
// flag; the roles stop issuing work, wait (bounded) for their copies and MMAs
// in flight, free the tensor memory and return.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"
#include "tc_common.cuh"

namespace convrot {

CONVROT_DEFINE_STATUS_WORD(status_word_gemm_tc)

namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;           // fp16 elements per stage row = 128 bytes = one swizzle atom
constexpr int BK8 = 128;         // e4m3 elements per stage row (4-bit variant)
constexpr int KCHUNK = 1024;     // exact fp32 accumulation span of int8 codes (see above)
constexpr int KITER_PER_CHUNK = KCHUNK / BK;
// Stage rows per TMEM chunk. 4-bit codes: |q*q| <= 49, so a partial sum stays
// below 2^24 (exact in fp32) for any K up to 342 000 > CONVROT_MAX_K: one
// chunk per tile, drained once.
template <bool F8>
constexpr int kiter_per_chunk() { return F8 ? (1 << 30) : KITER_PER_CHUNK; }
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 32 * (2 + NUM_EPI_WARPS);
constexpr int TMEM_COLS = 512;
constexpr int GROUP_M = 16;
// Y leaves through TMA stores of 32 rows x 16 columns (one warp's rows),
// 32-byte swizzle: the 16-byte half of row r sits at half ^ (r >> 2 & 1).
constexpr int OUT_COLS = 16;
constexpr int OUT_PIECE_BYTES = 1024;
constexpr int OUT_BUFS = 2;      // output pieces in flight per epilogue warp

// CL = 1: one CTA computes a 128 x BN tile with cta_group::1 MMAs.
// CL = 2: a cluster pair computes a 256 x BN tile with cta_group::2 MMAs
// issued by the leader (rank 0); each CTA holds its own 128 A rows and half
// of the B tile (BN / 2 rows), and receives its 128 x BN half of D in its
// own tensor memory.
template <int BN, int CL>
struct Cfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_ROWS = BN / CL;  // rows of B held by one CTA
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int HALF = BN / 2;  // columns per epilogue thread
  // per epilogue warp: OUT_BUFS 32 x 16 bf16 output pieces for the tiled store
  static constexpr int OUT_BYTES = NUM_EPI_WARPS * OUT_BUFS * OUT_PIECE_BYTES;
  // per epilogue warp: the column scales and biases of its half tile
  static constexpr int EPI_BYTES = NUM_EPI_WARPS * HALF * 2 * 4;
  // as many stages as fit next to those, at most 200 KB of them
  static constexpr int STAGES_FIT = (232448 - 1024 - BAR_BYTES - OUT_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < (200 * 1024) / STAGE_BYTES ? STAGES_FIT : (200 * 1024) / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES + EPI_BYTES + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "the output pieces stay 1 KB aligned");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(HALF % 16 == 0, "the drain loads 32 or 16 columns at a time");
  // Instruction descriptor, kind::f16: D = F32 (bits 4-5 = 1), A = B = F16
  // (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
  // M >> 4 at bit 24.
  static constexpr uint32_t IDESC = idesc_f16(BM * CL, BN, false);
};

struct TcParams {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b[kMaxLinears];
  CUtensorMap tmap_y[kMaxLinears];  // Y [M, n] (bf16, or int32 when RAW) for the tiled stores (when y_tma)
  GemmOutputs outs;
  const float* sx;
  long long M;
  int K;
  int m_tiles;
  int n_tiles;
  int num_tiles;   // cluster tiles: (m tiles / cluster size, rounded up) x n tiles
  int y_tma;       // 1: Y through tmap_y; 0: direct stores
  int dp_tiles;    // tiles computed whole, round-robin over the clusters
  int sk_tiles;    // the tiles after those, each split along K ...
  int sk_pieces;   // ... into this many pieces, one per cluster
  int* ws_cnt;     // split tiles: arrival counter per 32-row slab
  int* ws_acc;     // split tiles: int32 sums, [tile][rank][warp][8-column chunk][lane][8]
  long long spin_limit;
};

// Wait for a phase, giving up after `limit` polls or when another role has
// aborted; returns false on give-up.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, long long limit,
                                              volatile int* abort_flag) {
  for (long long i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort_flag) return false;
    if (i > 128) __nanosleep(32);
  }
  return false;
}

// 16-byte global -> shared copy that reads `src_bytes` (0..16) bytes and
// zero-fills the rest; with src_bytes == 0 nothing is read.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void lds_128(uint32_t addr, float* v) {
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr));
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag) {
  *abort_flag = 1;
  record_status(CONVROT_ERR_TIMEOUT);
}

// Cluster tile t -> (m block of this CTA, n tile). The CL CTAs of a cluster
// take CL adjacent m blocks of the same n tile (they share its B tile).
template <int CL>
__device__ __forceinline__ void decode_tile(const TcParams& p, int t, int rank, int& m_blk, int& n_glob, int& li,
                                            int& n_local) {
  const int m_pairs = (p.m_tiles + CL - 1) / CL;
  const int per_group = GROUP_M * p.n_tiles;
  const int g = t / per_group;
  const int first_m = g * GROUP_M;
  const int gm = min(m_pairs - first_m, GROUP_M);
  const int r = t - g * per_group;
  m_blk = (first_m + r % gm) * CL + rank;
  n_glob = r / gm;
  li = 0;
  while (li + 1 < p.outs.count && n_glob >= p.outs.o[li + 1].tile_begin) ++li;
  n_local = n_glob - p.outs.o[li].tile_begin;
}

// Work item i of cluster c (of nc): tile t over k blocks [kb0, kb1); piece
// is -1 for a whole tile, else the index of the K piece of a split tile.
// Returns false past the cluster's last item.
// With a split, dp_tiles is a multiple of nc: every cluster has dp_tiles / nc
// whole tiles and at most one piece. The piece comes first: its reduction,
// and the epilogue of the last piece of each tile, then overlap the MMAs of
// the whole tiles instead of trailing them.
__device__ __forceinline__ bool work_item(const TcParams& p, int c, int nc, int i, int nk, int& t, int& kb0, int& kb1,
                                         int& piece) {
  const bool has_piece = p.sk_tiles != 0 && c < p.sk_tiles * p.sk_pieces;
  if (has_piece && i == 0) {
    t = p.dp_tiles + c / p.sk_pieces;
    piece = c % p.sk_pieces;
    kb0 = piece * nk / p.sk_pieces;
    kb1 = (piece + 1) * nk / p.sk_pieces;
    return true;
  }
  const int td = c + (has_piece ? i - 1 : i) * nc;
  if (td >= p.dp_tiles) return false;
  t = td;
  kb0 = 0;
  kb1 = nk;
  piece = -1;
  return true;
}

template <int BN, bool RAW, int CL, bool F8>
__global__ void __launch_bounds__(THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<BN, CL>;
  static_assert(CL == 1 || CL == 2, "cluster of 1 or 2 CTAs");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* out_smem = smem + C::STAGES * C::STAGE_BYTES;  // 1 KB aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(out_smem + C::OUT_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* final_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned char* epi_smem = out_smem + C::OUT_BYTES + C::BAR_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int BKE = F8 ? BK8 : BK;  // K values per 128-byte stage row
  const int nk = p.K / BKE;
  const int rank = CL == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster_id = blockIdx.x / CL, nclusters = gridDim.x / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // released by the (leader's) MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], NUM_EPI_WARPS * CL);  // the epilogue warps of every CTA of the pair
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (CL == 1) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer may multicast into this CTA's buffers only after its barriers exist
  if constexpr (CL > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent of the previous kernel in the stream
  // (the rotate+quantize that writes A and s_x): the set-up above and the
  // first round of weight tiles overlap its last CTAs. The producer (before
  // its first A tile) and the epilogue (before s_x) wait for that grid to
  // complete and flush (griddepcontrol.wait); the MMA issuer reads only
  // shared memory.
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int armed_round[C::STAGES];
      for (int s = 0; s < C::STAGES; ++s) armed_round[s] = -1;
      // the weights do not depend on the previous kernel: request the first
      // round's B tiles (and arm those stages) before waiting for it
      auto load_b = [&](int s, int kb, int li, int n_local) {
        const uint32_t sb = smem_base + s * C::STAGE_BYTES + C::A_BYTES;
        if constexpr (CL == 1) {
          mbar_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(sb, &p.tmap_b[li], kb * BKE, n_local * BN, &full[s]);
        } else {
          // both CTAs' bytes complete on the leader's barrier, which the
          // leader arms for the pair
          if (rank == 0) mbar_expect_tx(&full[s], CL * C::STAGE_BYTES);
          tma_load_2d_pair(sb, &p.tmap_b[li], kb * BKE, n_local * BN + rank * C::B_ROWS, mapa_shared(&full[s], 0));
        }
      };
      auto load_a = [&](int s, int kb, int m_blk) {
        const uint32_t sa = smem_base + s * C::STAGE_BYTES;
        if constexpr (CL == 1) {
          tma_load_2d(sa, &p.tmap_a, kb * BKE, m_blk * BM, &full[s]);
        } else {
          tma_load_2d_pair(sa, &p.tmap_a, kb * BKE, m_blk * BM, mapa_shared(&full[s], 0));
        }
      };
      int t, kb0, kb1, pc;
      {
        int it0 = 0;
        for (int i = 0; it0 < C::STAGES && work_item(p, cluster_id, nclusters, i, nk, t, kb0, kb1, pc); ++i) {
          int m_blk, n_glob, li, n_local;
          decode_tile<CL>(p, t, rank, m_blk, n_glob, li, n_local);
          for (int kb = kb0; kb < kb1 && it0 < C::STAGES; ++kb, ++it0) load_b(it0, kb, li, n_local);
        }
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && work_item(p, cluster_id, nclusters, i, nk, t, kb0, kb1, pc); ++i) {
        int m_blk, n_glob, li, n_local;
        decode_tile<CL>(p, t, rank, m_blk, n_glob, li, n_local);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES, round = it / C::STAGES;
          if (round > 0) {
            if (!wait_or_abort(&empty[s], (round & 1) ^ 1, p.spin_limit, abort_flag)) {
              raise_abort(abort_flag);
              ok = false;
              break;
            }
            load_b(s, kb, li, n_local);
          }
          load_a(s, kb, m_blk);
          armed_round[s] = round;
        }
      }
      // every armed copy must have landed before the CTA may exit (in a pair
      // the leader's barriers count both CTAs' copies; the closing cluster
      // barrier holds the peer until the leader has seen them)
      if (CL == 1 || rank == 0)
        for (int s = 0; s < C::STAGES; ++s)
          if (armed_round[s] >= 0 && !mbar_wait_bounded(&full[s], armed_round[s] & 1, p.spin_limit))
            raise_abort(abort_flag);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && CL == 2 && rank != 0) {
      // the peer issues nothing; its half of D is complete when the leader's
      // final commit arrives here
      if (!mbar_wait_bounded(final_bar, 0, p.spin_limit)) raise_abort(abort_flag);
    } else if (lane == 0) {
      int it = 0, chunk = 0;
      bool ok = true;
      int t, kb0, kb1, pc;
      for (int i = 0; ok && work_item(p, cluster_id, nclusters, i, nk, t, kb0, kb1, pc); ++i) {
        for (int kb = kb0; kb < kb1 && ok;) {
          const int b = chunk & 1, u = chunk >> 1;
          if (!wait_or_abort(&acc_empty[b], (u & 1) ^ 1, p.spin_limit, abort_flag)) {
            raise_abort(abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
          const int kend = min(kb + kiter_per_chunk<F8>(), kb1);
          const int kstart = kb;
          for (; kb < kend; ++kb, ++it) {
            const int s = it % C::STAGES, round = it / C::STAGES;
            if (!wait_or_abort(&full[s], round & 1, p.spin_limit, abort_flag)) {
              raise_abort(abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_base + s * C::STAGE_BYTES;
            const uint32_t sb = sa + C::A_BYTES;
            // four MMAs per 128-byte row: K = 16 (fp16) or 32 (e4m3) each
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc = (kb != kstart || k > 0) ? 1u : 0u;
              if constexpr (CL == 1 && !F8) {
                tc_mma_f16(d_tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), C::IDESC, acc);
              } else if constexpr (CL == 1) {
                tc_mma_f8(d_tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), C::IDESC, acc);
              } else if constexpr (!F8) {
                tc_mma_f16_pair(d_tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), C::IDESC, acc);
              } else {
                tc_mma_f8_pair(d_tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), C::IDESC, acc);
              }
            }
            if constexpr (CL == 1) {
              tc_commit(&empty[s]);
            } else {
              tc_commit_pair_multicast(&empty[s], 3);
            }
          }
          if (!ok) break;
          if constexpr (CL == 1) {
            tc_commit(&acc_full[b]);
          } else {
            tc_commit_pair_multicast(&acc_full[b], 3);
          }
          ++chunk;
        }
      }
      // all issued MMAs complete before the tensor memory is released
      if constexpr (CL == 1) {
        tc_commit(final_bar);
      } else {
        tc_commit_pair_multicast(final_bar, 3);
      }
      if (!mbar_wait_bounded(final_bar, 0, p.spin_limit)) raise_abort(abort_flag);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    asm volatile("griddepcontrol.wait;" ::: "memory");  // s_x comes from the previous kernel
    const int q = warp & 3;              // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;    // which half of the BN columns
    const int row_in_tile = q * 32 + lane;
    const int col0 = half * C::HALF;
    // this warp's copy of the half tile's column scales, then biases
    const uint32_t wsw = smem_u32(epi_smem) + static_cast<uint32_t>((warp - 2) * C::HALF * 2 * 4);
    const uint32_t wbias = wsw + C::HALF * 4;
    const uint32_t wout = smem_u32(out_smem) + static_cast<uint32_t>((warp - 2) * OUT_BUFS * OUT_PIECE_BYTES);
    // this lane's row in an output piece, with the 32-byte swizzle
    const uint32_t out_row = static_cast<uint32_t>(lane) * 32;
    const uint32_t out_sw = static_cast<uint32_t>((lane >> 2) & 1) << 4;
    int ob = 0;  // output-buffer uses (tiled stores, bulk reductions) by this warp so far
    int chunk = 0;
    bool ok = true;
    int t, kb0, kb1, pc;
    for (int i = 0; ok && work_item(p, cluster_id, nclusters, i, nk, t, kb0, kb1, pc); ++i) {
      int m_blk, n_glob, li, n_local;
      decode_tile<CL>(p, t, rank, m_blk, n_glob, li, n_local);
      const int nch = (kb1 - kb0 + kiter_per_chunk<F8>() - 1) / kiter_per_chunk<F8>();
      const GemmOut& o = p.outs.o[li];
      const long long m = static_cast<long long>(m_blk) * BM + row_in_tile;
      const int nb = n_local * BN + col0;
      float srow = 0.0f;
      if constexpr (!RAW) {
        __syncwarp();  // every lane has read the previous tile's values
        // fetched now, used after the last chunk: the loads overlap the MMAs.
        // Columns past N read as zero (the warp's previous reads of these
        // buffers finished before its final stores of the previous tile).
        if (m < p.M) srow = __ldg(p.sx + m);
        for (int j = 4 * lane; j < C::HALF; j += 128) {
          const int n = nb + j;
          const int bytes = n < o.n ? 4 * min(4, o.n - n) : 0;
          cp_async_16(wsw + 4 * j, bytes ? static_cast<const void*>(o.sw + n) : static_cast<const void*>(o.sw), bytes);
          const int bb = o.bias ? bytes : 0;
          cp_async_16(wbias + 4 * j, bb ? static_cast<const void*>(o.bias + n) : static_cast<const void*>(o.sw), bb);
        }
        cp_async_commit();
      }
      int acc[C::HALF];
#pragma unroll
      for (int j = 0; j < C::HALF; ++j) acc[j] = 0;
      for (int c = 0; c < nch; ++c, ++chunk) {
        const int b = chunk & 1, u = chunk >> 1;
        // every lane waits; the warp proceeds only if all lanes saw the phase
        // (the TMEM loads below are warp-collective)
        const bool got = wait_or_abort(&acc_full[b], u & 1, p.spin_limit, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) raise_abort(abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN + col0);
#pragma unroll
        for (int j = 0; j < C::HALF / 32; ++j) {
          uint32_t r[32];
          tc_ld_32x32b_x32(taddr + j * 32, r);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[j * 32 + e] += __float2int_rz(__uint_as_float(r[e]));
        }
        if constexpr (C::HALF % 32 == 16) {  // e.g. BN = 224: 112 columns = 3 x 32 + 16
          constexpr int j0 = C::HALF - 16;
          uint32_t r[16];
          tc_ld_32x32b_x16(taddr + j0, r);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[j0 + e] += __float2int_rz(__uint_as_float(r[e]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CL == 1 || rank == 0) {
            mbar_arrive(&acc_empty[b]);
          } else {
            mbar_arrive_cluster(mapa_shared(&acc_empty[b], 0));  // the leader reuses the buffer
          }
        }
      }
      if (!ok) break;

      if constexpr (!RAW) {
        cp_async_wait_all();
        __syncwarp();
      }
      if (pc >= 0) {
        // a piece of a split tile: add this warp's 32-row slab of partial sums
        // into the tile's workspace slot by bulk reductions in L2 (8 columns
        // = 1 KB at a time, staged in the output buffers). The warp whose
        // piece arrives last for the slab reads the totals, clears the slot
        // and the counter for the next call, and finishes the slab; the
        // others move on.
        const int slab = ((t - p.dp_tiles) * CL + rank) * NUM_EPI_WARPS + (warp - 2);
        int* wslab = p.ws_acc + static_cast<long long>(slab) * (C::HALF * 32);  // [8-column chunk][lane][8]
#pragma unroll
        for (int j = 0; j < C::HALF; j += 8) {
          const uint32_t pb = wout + static_cast<uint32_t>((ob % OUT_BUFS) * OUT_PIECE_BYTES);
          if (ob >= OUT_BUFS) {
            if (lane == 0) bulk_wait_read<OUT_BUFS - 1>();
            __syncwarp();
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + lane * 32), "r"(acc[j]), "r"(acc[j + 1]),
                       "r"(acc[j + 2]), "r"(acc[j + 3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + lane * 32 + 16), "r"(acc[j + 4]),
                       "r"(acc[j + 5]), "r"(acc[j + 6]), "r"(acc[j + 7])
                       : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_reduce_add_s32(wslab + j * 32, pb, OUT_PIECE_BYTES);
            bulk_commit();
          }
          ++ob;
        }
        int prev = 0;
        if (lane == 0) {
          bulk_wait_all();  // the additions are complete ...
          fence_proxy_async_global();
          __threadfence();  // ... and visible before the arrival is counted
          prev = atomicAdd(p.ws_cnt + slab, 1);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != p.sk_pieces - 1) continue;
        __threadfence();
        fence_proxy_async_global();
#pragma unroll
        for (int j = 0; j < C::HALF; j += 8) {
          const int4 lo = __ldcg(reinterpret_cast<const int4*>(wslab + j * 32 + lane * 8));
          const int4 hi = __ldcg(reinterpret_cast<const int4*>(wslab + j * 32 + lane * 8 + 4));
          acc[j] = lo.x; acc[j + 1] = lo.y; acc[j + 2] = lo.z; acc[j + 3] = lo.w;
          acc[j + 4] = hi.x; acc[j + 5] = hi.y; acc[j + 6] = hi.z; acc[j + 7] = hi.w;
        }
#pragma unroll
        for (int j = 0; j < C::HALF; j += 8) {
          __stcg(reinterpret_cast<int4*>(wslab + j * 32 + lane * 8), make_int4(0, 0, 0, 0));
          __stcg(reinterpret_cast<int4*>(wslab + j * 32 + lane * 8 + 4), make_int4(0, 0, 0, 0));
        }
        if (lane == 0) atomicExch(p.ws_cnt + slab, 0);
      }
      if (RAW && p.y_tma) {
        // raw accumulators: the warp's 32 rows x HALF columns leave in 32 x 8
        // int32 pieces (32 bytes a row, the bf16 pieces' layout), through the
        // same two buffers; rows past M and columns past n are clipped
        const int row0 = m_blk * BM + q * 32;
        const bool rows_in = row0 < p.M;
#pragma unroll
        for (int j = 0; j < C::HALF; j += 8) {
          if (!rows_in || nb + j >= o.n) continue;  // warp-uniform
          const uint32_t pb = wout + static_cast<uint32_t>((ob % OUT_BUFS) * OUT_PIECE_BYTES);
          if (ob >= OUT_BUFS) {
            if (lane == 0) bulk_wait_read<OUT_BUFS - 1>();
            __syncwarp();
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + out_row + out_sw), "r"(acc[j]),
                       "r"(acc[j + 1]), "r"(acc[j + 2]), "r"(acc[j + 3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + out_row + (16u ^ out_sw)), "r"(acc[j + 4]),
                       "r"(acc[j + 5]), "r"(acc[j + 6]), "r"(acc[j + 7])
                       : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmap_y[li], pb, nb + j, row0);
            bulk_commit();
          }
          ++ob;
        }
      } else if (!RAW && p.y_tma) {
        // The warp's 32 rows x HALF columns leave in 32 x 16 pieces through
        // two buffers; lane 0 issues the stores and, before a buffer is
        // rewritten, waits until the copy issued from it two uses ago has
        // read it. Rows past M and columns past n are clipped by the copy.
        const int row0 = m_blk * BM + q * 32;
        const bool rows_in = row0 < p.M;
#pragma unroll
        for (int j = 0; j < C::HALF; j += OUT_COLS) {
          if (!rows_in || nb + j >= o.n) continue;  // warp-uniform
          const uint32_t pb = wout + static_cast<uint32_t>((ob % OUT_BUFS) * OUT_PIECE_BYTES);
          if (ob >= OUT_BUFS) {
            if (lane == 0) bulk_wait_read<OUT_BUFS - 1>();
            __syncwarp();
          }
          uint32_t w[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float swv[8], bv[8];
            lds_128(wsw + 4 * (j + 8 * h), swv);
            lds_128(wsw + 4 * (j + 8 * h) + 16, swv + 4);
            lds_128(wbias + 4 * (j + 8 * h), bv);
            lds_128(wbias + 4 * (j + 8 * h) + 16, bv + 4);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int c = j + 8 * h + e;
              const float y0 = fmaf(static_cast<float>(acc[c]), srow * swv[e], bv[e]);
              const float y1 = fmaf(static_cast<float>(acc[c + 1]), srow * swv[e + 1], bv[e + 1]);
              const __nv_bfloat162 hv = __floats2bfloat162_rn(y0, y1);
              w[4 * h + e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
            }
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + out_row + out_sw), "r"(w[0]), "r"(w[1]),
                       "r"(w[2]), "r"(w[3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + out_row + (16u ^ out_sw)), "r"(w[4]),
                       "r"(w[5]), "r"(w[6]), "r"(w[7])
                       : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmap_y[li], pb, nb + j, row0);
            bulk_commit();
          }
          ++ob;
        }
      } else if (m < p.M) {
        if constexpr (RAW) {
          int* yrow = static_cast<int*>(o.y) + m * o.ldy;
#pragma unroll
          for (int j = 0; j < C::HALF; j += 4) {
            const int n = nb + j;
            if (n + 4 <= o.n) {
              *reinterpret_cast<int4*>(yrow + n) = make_int4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (n + e < o.n) yrow[n + e] = acc[j + e];
            }
          }
        } else {
          __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(o.y) + m * o.ldy;
#pragma unroll
          for (int j = 0; j < C::HALF; j += 8) {
            const int n = nb + j;
            // 8 scales and 8 biases, the same address in every lane (broadcast)
            float swv[8], bv[8];
            lds_128(wsw + 4 * j, swv);
            lds_128(wsw + 4 * j + 16, swv + 4);
            lds_128(wbias + 4 * j, bv);
            lds_128(wbias + 4 * j + 16, bv + 4);
            if (n + 8 <= o.n) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const float y0 = fmaf(static_cast<float>(acc[j + e]), srow * swv[e], bv[e]);
                const float y1 = fmaf(static_cast<float>(acc[j + e + 1]), srow * swv[e + 1], bv[e + 1]);
                const __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
                w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
              }
              stg_128(yrow + n, make_uint4(w[0], w[1], w[2], w[3]));
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (n + e < o.n) yrow[n + e] = __float2bfloat16_rn(fmaf(static_cast<float>(acc[j + e]), srow * swv[e], bv[e]));
            }
          }
        }
      }
    }
  }

  cp_async_wait_all();  // no copy into shared memory outlives the CTA (abort path)
  if (warp >= 2 && (threadIdx.x & 31) == 0) bulk_wait_all();  // the tiled stores are complete
  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still write into it
  if constexpr (CL > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CL == 1) {
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    } else {
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    }
  }
}

// ---- host -------------------------------------------------------------------

// Operand map: [rows][K] fp16 (or e4m3 bytes), boxes of 128 bytes x box_rows.
bool make_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, long long rows, int K, int box_rows, bool f8) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * (f8 ? 1 : 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(f8 ? BK8 : BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// Column tile width. One MMA reads 4 KB of A per SM whatever N is, plus
// N * 16 bytes of B, while it does 128 * N * 32 flops per SM; at ~64 bytes of
// operand reads per cycle and 8192 flops per cycle the cycles per MMA are
// max(N / 2, (4096 + 16 N) / 64), so narrow tiles run the tensor cores below
// peak (measured on GB300, 2-SM MMA: N = 256 / 192 / 128 reach 0.85 / 0.71 /
// 0.50 of the bf16 peak on the same shapes; 128 is therefore not offered).
// The choice minimizes
// rounds x (time of one tile), a round being one tile per resident cluster;
// a last round split along K costs 1 / pieces of a round plus a fixed time
// for the partial sums' trip through L2 and the exposed final epilogue
// (about 10 us measured on GB300; in the model's cycles, with the tensor
// pipes at the ~72 % they sustain here, some 15000).
double mma_cycles_per_column(int bn) {
  const double compute = bn / 2.0;
  const double operands = (4096.0 + 16.0 * bn) / 64.0;
  return std::max(compute, operands) / bn;
}

// Workspace layout: arrival counters in the first 4 KB, then the partial sums.
constexpr long long kWsCounterBytes = 4096;

struct SplitPlan {
  int dp_tiles;  // whole tiles
  int sk_tiles;  // split tiles (0: no split)
  int pieces;    // K pieces per split tile
};

// Split the last round along K when it would leave at least half of the
// clusters idle and the workspace has a slot for every split tile; each
// piece keeps at least two k blocks.
SplitPlan plan_split(long long tiles, int clusters, int nk, int bn, int cl, long long ws_bytes) {
  SplitPlan sp{static_cast<int>(tiles), 0, 1};
  if (ws_bytes <= kWsCounterBytes || clusters < 2) return sp;
  // one slot of sums per split tile, one counter per 32-row slab
  const long long slot_bytes = static_cast<long long>(cl) * BM * bn * 4;
  const long long slots = (ws_bytes - kWsCounterBytes) / slot_bytes;
  const long long tail = tiles % clusters;
  if (tail == 0 || tail > slots || tail * cl * NUM_EPI_WARPS * 4 > kWsCounterBytes) return sp;
  const long long pieces = std::min<long long>(clusters / tail, nk / 2);
  if (pieces < 2) return sp;
  sp.dp_tiles = static_cast<int>(tiles - tail);
  sp.sk_tiles = static_cast<int>(tail);
  sp.pieces = static_cast<int>(pieces);
  return sp;
}

constexpr double kSplitOverheadCycles = 15000.0;

// Candidate tile widths, and for each the clusters resident at once.
constexpr int kBnCandidates[3] = {256, 224, 192};

int choose_bn(long long M, int K, int bke, const GemmOutputs& outs, const int (&resident)[3], int cl,
              long long ws_bytes) {
  const long long mt = ((M + BM - 1) / BM + cl - 1) / cl;
  int best = 256;
  double best_cost = -1.0;
  for (int c = 0; c < 3; ++c) {
    const int bn = kBnCandidates[c];
    const int clusters = std::max(1, resident[c]);
    long long nt = 0;
    for (int i = 0; i < outs.count; ++i) nt += (outs.o[i].n + bn - 1) / bn;
    const long long tiles = mt * nt;
    const SplitPlan sp = plan_split(tiles, clusters, K / bke, bn, cl, ws_bytes);
    // cycles of one tile: k blocks x MMAs per block x their cycles
    const double tile = static_cast<double>(K / bke) * 4 * bn * mma_cycles_per_column(bn);
    const double cost = sp.sk_tiles ? (sp.dp_tiles / clusters + 1.0 / sp.pieces) * tile + kSplitOverheadCycles
                                    : static_cast<double>((tiles + clusters - 1) / clusters) * tile;
    if (best_cost < 0 || cost < best_cost * 0.999) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Clusters of this instantiation that can be resident at once (one CTA per
// SM without pairs); also sets the kernel's shared-memory limit.
template <int BN, bool RAW, int CL, bool F8>
cudaError_t resident_clusters(int sms, int* out) {
  using C = Cfg<BN, CL>;
  auto kern = gemm_tc_kernel<BN, RAW, CL, F8>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  *out = sms;
  if constexpr (CL > 1) {
    e = max_active_clusters(reinterpret_cast<const void*>(kern), THREADS, C::SMEM, CL, out);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BN, bool RAW, int CL, bool F8>
cudaError_t launch_bn(EncodeTiledFn enc, const void* Qx16, const float* sx, long long M, int K, GemmOutputs outs,
                      void* ws, long long ws_bytes, cudaStream_t st, int sms) {
  using C = Cfg<BN, CL>;
  constexpr int BKE = F8 ? BK8 : BK;
  TcParams p;
  memset(&p, 0, sizeof(p));
  if (!make_map(enc, &p.tmap_a, Qx16, M, K, BM, F8)) return cudaErrorInvalidValue;
  int nt = 0;
  for (int i = 0; i < outs.count; ++i) {
    outs.o[i].tile_begin = nt;
    nt += (outs.o[i].n + BN - 1) / BN;
    // in a pair each CTA loads its BN / 2 rows of the B tile
    if (!make_map(enc, &p.tmap_b[i], outs.o[i].qw16, outs.o[i].n, K, BN / CL, F8)) return cudaErrorInvalidValue;
  }
  // Y through tiled stores when every output allows it: 16-byte aligned base
  // and row pitch, at least one full piece wide. A piece is 32 rows of 32
  // bytes: 16 bf16 columns, or 8 int32 columns of raw accumulators.
  constexpr int y_bytes = RAW ? 4 : 2;
  constexpr int piece_cols = 32 / y_bytes;
  p.y_tma = 1;
  for (int i = 0; i < outs.count && p.y_tma; ++i) {
    const GemmOut& o = outs.o[i];
    if (reinterpret_cast<uintptr_t>(o.y) % 16 != 0 || (o.ldy * y_bytes) % 16 != 0 || o.n < piece_cols || M < 32) {
      p.y_tma = 0;
      break;
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(o.n), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(o.ldy) * y_bytes};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(piece_cols), 32};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&p.tmap_y[i], RAW ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.y, dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      p.y_tma = 0;
  }
  p.outs = outs;
  p.sx = sx;
  p.M = M;
  p.K = K;
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  p.n_tiles = nt;
  const long long tiles = static_cast<long long>((p.m_tiles + CL - 1) / CL) * nt;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.num_tiles = static_cast<int>(tiles);
  p.spin_limit = kDefaultSpinLimit;
  auto kern = gemm_tc_kernel<BN, RAW, CL, F8>;
  // clusters that are resident together (the count the tile width was chosen
  // under): the split plan needs the real count
  int clusters = 0;
  cudaError_t e = resident_clusters<BN, RAW, CL, F8>(sms, &clusters);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const SplitPlan sp = plan_split(tiles, clusters, K / BKE, BN, CL, ws ? ws_bytes : 0);
  // oversize guard: the split's counters and sums must fit the workspace
  if (sp.sk_tiles && kWsCounterBytes + static_cast<long long>(sp.sk_tiles) * CL * BM * BN * 4 > ws_bytes)
    return cudaErrorInvalidValue;
  p.dp_tiles = sp.dp_tiles;
  p.sk_tiles = sp.sk_tiles;
  p.sk_pieces = sp.pieces;
  p.ws_cnt = static_cast<int*>(ws);
  p.ws_acc = ws ? reinterpret_cast<int*>(static_cast<char*>(ws) + kWsCounterBytes) : nullptr;
  // a split runs on every cluster (its whole tiles are a multiple of them)
  const int nc = sp.sk_tiles ? clusters : static_cast<int>(std::min<long long>(tiles, clusters));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * nc);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  // may start while the previous kernel of the stream finishes (the kernel
  // waits for it with griddepcontrol.wait before touching its outputs)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool RAW, int CL, bool F8>
cudaError_t launch_cl(EncodeTiledFn enc, const void* Qx16, const float* sx, long long M, int K,
                      const GemmOutputs& outs, void* ws, long long ws_bytes, cudaStream_t st, int sms) {
  int resident[3];
  cudaError_t e = resident_clusters<256, RAW, CL, F8>(sms, &resident[0]);
  if (e == cudaSuccess) e = resident_clusters<224, RAW, CL, F8>(sms, &resident[1]);
  if (e == cudaSuccess) e = resident_clusters<192, RAW, CL, F8>(sms, &resident[2]);
  if (e != cudaSuccess) return e;
  switch (choose_bn(M, K, F8 ? BK8 : BK, outs, resident, CL, ws ? ws_bytes : 0)) {
    case 256: return launch_bn<256, RAW, CL, F8>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
    case 224: return launch_bn<224, RAW, CL, F8>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
    default: return launch_bn<192, RAW, CL, F8>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
  }
}

}  // namespace

bool gemm_tc_supported(long long M, int K) { return M > 64 && K % BK == 0 && K >= BK; }

// Qx16: fp16 codes, or with f8 the e4m3 codes of the 4-bit variant (any M;
// K a multiple of 128; the outputs' qw16 point at e4m3 weights).
cudaError_t gemm_tc_launch(const void* Qx16, const float* sx, long long M, int K, const GemmOutputs& outs, bool raw,
                           bool f8, void* ws, long long ws_bytes, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (K % (f8 ? BK8 : BK) != 0) return cudaErrorInvalidValue;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const int sms = device_sm_count();
  // CTA pairs run the 2-SM MMA when there are at least two row blocks
  if (f8) {
    if (M > BM)
      return raw ? launch_cl<true, 2, true>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms)
                 : launch_cl<false, 2, true>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
    return raw ? launch_cl<true, 1, true>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms)
               : launch_cl<false, 1, true>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
  }
  if (M > BM)
    return raw ? launch_cl<true, 2, false>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms)
               : launch_cl<false, 2, false>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
  return raw ? launch_cl<true, 1, false>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms)
             : launch_cl<false, 1, false>(enc, Qx16, sx, M, K, outs, ws, ws_bytes, st, sms);
}

// The schedule gemm_tc_launch picks, computed on the host alone: tile width,
// whole tiles, and the tiles of the last round split along K with their
// piece count. It takes one cluster resident per SM pair (per SM without
// pairs), which is what the kernel's shared memory allows; the launch takes
// the count from the occupancy query, so the two agree whenever that query
// returns sms / cl.
bool gemm_tc_plan(long long M, int K, const GemmOutputs& outs, bool f8, int sms, long long ws_bytes, int* bn,
                  long long* whole, long long* split, int* pieces) {
  const int bke = f8 ? BK8 : BK;
  if (M <= 0 || K < bke || K % bke != 0 || sms < 1 || outs.count < 1) return false;
  const int cl = M > BM ? 2 : 1;
  const int per = std::max(1, sms / cl);
  const int resident[3] = {per, per, per};
  const int b = choose_bn(M, K, bke, outs, resident, cl, ws_bytes);
  long long nt = 0;
  for (int i = 0; i < outs.count; ++i) nt += (outs.o[i].n + b - 1) / b;
  const long long tiles = ((M + BM - 1) / BM + cl - 1) / cl * nt;
  if (tiles > 0x7fffffffLL) return false;  // the launch rejects such a grid too
  const SplitPlan sp = plan_split(tiles, per, K / bke, b, cl, ws_bytes);
  *bn = b;
  *whole = sp.dp_tiles;
  *split = sp.sk_tiles;
  *pieces = sp.pieces;
  return true;
}

}  // namespace convrot
