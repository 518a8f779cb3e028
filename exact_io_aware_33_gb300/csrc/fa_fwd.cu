// Forward pass of exact attention on sm_103a.
//
// Method ("Flash Attention: IO-Aware Exact Attention", sections "Online
// softmax makes tiling exact" and "Loop order changes which data is
// reloaded"): a block of query rows stays on chip with its row state while
// every key/value tile streams past; per row the kernel carries a running
// maximum m, a denominator l and an unnormalised numerator a, rescales the
// old sums by alpha = exp(m_old - m_new) when the maximum moves, and divides
// once at the end. Scores S and probabilities P exist only in tensor memory.
//
// CTA organisation (320 threads, one CTA per SM):
//   warps 0-3  softmax warpgroup of query tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax warpgroup of query tile 1
//   warp  8    tcgen05 MMA issue (one elected lane) and TMEM allocation
//   warp  9    TMA producer (one thread)
// Every warp keeps the launch allocation (168 registers): lowering the MMA
// warp's budget slows its issue loop, and the tensor core's issue queue is
// only a few instructions deep, so that shows directly in the step time.
// Each CTA owns 256 query rows of one (batch, head): two 128-row tiles that
// ping-pong, so the tensor core works on one tile's QK^T / PV while the
// other tile's softmax runs. The one-tile form (QT = 1; 192 threads) is used
// at d = d_v = 64, two CTAs per SM, and at d = d_v = 256, where a tile's S
// (128 columns) and O (256 columns) fill the tensor memory and its Q, K and
// V tiles (64 KiB each, a single K/V stage) the shared memory.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128)  S of tile 0; its first 64 columns are overwritten by P (bf16
//              pairs) which the P.V MMA reads straight from TMEM
//   [128,256)  S / P of tile 1
//   [256,256+d)      O accumulator of tile 0
//   [256+d,256+2d)   O accumulator of tile 1
//
// Shared memory: Q tiles (2 x 128 x d bf16), and rings of K and V tiles
// (stages x 128 x d bf16 each), all in the 128-byte-swizzled layout TMA
// writes and the tensor core reads; d = 128 (256) is stored as two (four)
// 64-column chunks. The online-softmax statistics never leave registers.
//
// Exactness note: the reference maximum of a row only moves when a tile's
// maximum exceeds it by more than 2^8 in the exponent (log2 units); until
// then exp2(s - m_ref) <= 256 is summed as is. Final division and LSE use
// the same m_ref, so the result is the same function -- only rounding
// changes.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

// D: head size of Q and K; DV: head size of V and O; QT: 128-row query tiles
// per CTA. QT = 2 shares each K/V tile between two query tiles; QT = 1 (used
// at d = d_v = 64) needs half the tensor memory and shared memory, so two
// CTAs share an SM and one's start-up and write-back overlap the other's
// key loop.
template <int D, int DV, int QT = 2>
struct FwdCfg {
  static constexpr int kQTiles = QT;
  static constexpr int kSoftmaxThreads = 128 * QT;
  static constexpr int kMmaWarp = kSoftmaxThreads / 32;
  static constexpr int kLoadWarp = kMmaWarp + 1;
  static constexpr int kThreads = kSoftmaxThreads + 64;  // + the MMA warp and the TMA warp
  // two CTAs per SM for the one-tile form at d = d_v = 64; d = d_v = 256
  // (one tile, 192 KiB of tiles) fills the SM alone
  static constexpr int kCtasPerSm = (QT == 1 && D + DV <= 128) ? 2 : 1;
  static constexpr int kChunks = D / 64;
  static constexpr int kChunksV = DV / 64;
  static constexpr int kChunkBytes = kBlockM * 64 * 2;        // 16 KiB
  static constexpr int kTileBytes = kChunks * kChunkBytes;    // 128 rows x d (Q, K)
  static constexpr int kVTileBytes = kChunksV * kChunkBytes;  // 128 rows x d_v (V)
  // K/V ring depth: as many stages as fit next to the Q tiles (QT = 1 at
  // d = 64: two CTAs per SM; at d = 256 a 64 KiB Q tile and one 64 KiB K
  // and V tile each fill the shared memory)
  static constexpr int kStages =
      QT == 1 ? (D + DV <= 128 ? 2 : 1) : (D == 64 && DV == 64) ? 4 : (D + DV == 192 ? 3 : 2);
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kVTileBytes;
  // barrier indices
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;
  static constexpr int kBarKEmpty = kBarKFull + kStages;
  static constexpr int kBarVFull = kBarKEmpty + kStages;
  static constexpr int kBarVEmpty = kBarVFull + kStages;
  static constexpr int kBarSFull = kBarVEmpty + kStages;
  static constexpr int kBarPFull = kBarSFull + kQTiles;
  static constexpr int kBarOFinal = kBarPFull + kQTiles;
  static constexpr int kBarSFree = kBarOFinal + kQTiles;   // separate-P layout only
  static constexpr int kBarPVDone = kBarSFree + kQTiles;   // separate-P layout only
  static constexpr int kBarDrain = kBarPVDone + kQTiles;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base
  static constexpr uint32_t kColO = 128 * QT;
  // With d_v = 64 the two S tiles and two O accumulators take 384 columns,
  // so each tile's P gets 64 columns of its own at kColP: the softmax
  // releases S as soon as it has loaded it and the next tile's QK^T
  // overlaps the exponentials. With d_v = 128 (or 256) the columns are full
  // and P overwrites S.
  static constexpr bool kSepP = (DV == 64);
  static constexpr uint32_t kColP = kColO + QT * DV;
  // S, O (and P) of every tile, rounded up to a power of two for the allocation
  static constexpr uint32_t kColsUsed = kColP + (kSepP ? QT * 64 : 0);
  static constexpr uint32_t kTmemCols = kColsUsed <= 256 ? 256 : 512;
  static_assert(kColsUsed <= 512, "forward accumulators exceed tensor memory");
  static_assert(kSmemBytes <= 232448, "forward tiles exceed shared memory");
};

struct FwdArgs {
  __nv_bfloat16* o;    // [BH, Nq, D] (whole-range launch)
  float* lse;          // [BH, Nq]
  float* part_o;       // [splits, BH, Nq, D] fp32 normalised partial outputs (split launch)
  float* part_lse;     // [splits, BH, Nq] natural-log partial LSE (split launch)
  int* status;
  int Nq, Nk;
  int kv_off;          // Nk - Nq: causal query i sits at key position i + kv_off
  int window;          // 0 = none; else keys j <= i + kv_off - window are masked
  int BH;
  int causal;
  int num_pairs;
  int split_tiles;     // key tiles per split (all of them when not split)
  int split_mode;      // 1: write fp32 partial states instead of O / LSE
  float scale_log2;    // scale * log2(e), > 0
  Dropout drop;        // kDrop kernels only
};

// kDrop: dropout on the probabilities that multiply V (see Dropout); the
// row sums and the LSE are those of the softmax itself.
template <int D, int DV, int QT, bool kDrop>
__global__ void __launch_bounds__(FwdCfg<D, DV, QT>::kThreads, FwdCfg<D, DV, QT>::kCtasPerSm)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<D, DV, QT>;
  constexpr int kQTiles = C::kQTiles;
  constexpr int kMmaWarp = C::kMmaWarp;
  constexpr int kLoadWarp = C::kLoadWarp;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kMiscOff + 4);

  // Key tiles each query tile needs: the causal limit (keys up to the last
  // row's position), the window (keys after the first row's position minus
  // the window), and this CTA's split of the key range. The CTA streams the
  // union [j_first, j_first + n_stream) of its two tiles' ranges once; tile
  // t takes part in stream steps [a_t, a_t + n_t).
  const int Nq = args.Nq, Nk = args.Nk;
  const int bh = blockIdx.x % args.BH;
  const int pair = args.num_pairs - 1 - static_cast<int>(blockIdx.x / args.BH);
  const int n_kv = (Nk + kBlockN - 1) / kBlockN;
  const int split_lo = blockIdx.y * args.split_tiles;
  const int split_hi = min(n_kv, split_lo + args.split_tiles);
  int q_row0[kQTiles], lo_t[kQTiles], n_t[kQTiles];
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    q_row0[t] = pair * (kBlockM * kQTiles) + t * kBlockM;
    int lo = split_lo, hi = split_hi;
    if (args.causal) {
      const int last_row = min(q_row0[t] + kBlockM, Nq) - 1;
      hi = min(hi, (last_row + args.kv_off) / kBlockN + 1);
    }
    if (args.window) {
      const int first_key = q_row0[t] + args.kv_off - args.window + 1;
      if (first_key > 0) lo = max(lo, first_key / kBlockN);
    }
    lo_t[t] = lo;
    n_t[t] = (q_row0[t] >= Nq || hi <= lo) ? 0 : hi - lo;
  }
  int j_first = 0, j_end = 0;
  {
    bool any = false;
#pragma unroll
    for (int t = 0; t < kQTiles; ++t) {
      if (n_t[t] == 0) continue;
      if (!any || lo_t[t] < j_first) j_first = lo_t[t];
      if (!any || lo_t[t] + n_t[t] > j_end) j_end = lo_t[t] + n_t[t];
      any = true;
    }
  }
  const int n_stream = j_end - j_first;
  // stream steps [a_t, b_t) of each query tile (empty when n_t = 0)
  const int a0 = lo_t[0] - j_first, b0 = a0 + n_t[0];
  // (one query tile: tile "1" is empty)
  const int a1 = kQTiles > 1 ? lo_t[kQTiles - 1] - j_first : 0;
  const int b1 = kQTiles > 1 ? a1 + n_t[kQTiles - 1] : 0;

  const int warp = warp_id();
  const int lane = lane_id();
  int issued = 0;  // producer: K/V copies started (K of step jj is 2 jj, its V 2 jj + 1)

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQFull), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), 4);   // one arrival per softmax warp
      mbar_init(bar(C::kBarOFinal + t), 1);
      mbar_init(bar(C::kBarSFree + t), 4);
      mbar_init(bar(C::kBarPVDone + t), 1);
    }
    mbar_init(bar(C::kBarDrain), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();
  grid_dep_launch();

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      uint32_t q_bytes = 0;
#pragma unroll
      for (int t = 0; t < kQTiles; ++t)
        if (n_t[t] > 0) q_bytes += C::kTileBytes;
      mbar_arrive_expect_tx(bar(C::kBarQFull), q_bytes);
#pragma unroll
      for (int t = 0; t < kQTiles; ++t) {
        if (n_t[t] == 0) continue;
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(base + C::kQOff + t * C::kTileBytes + c * C::kChunkBytes, &tmQ,
                      bar(C::kBarQFull), c * 64, q_row0[t], bh);
      }
      bool ok = true;
      for (int jj = 0; jj < n_stream && ok; ++jj) {
        const int s = jj % C::kStages;
        const uint32_t ph = ((jj / C::kStages) + 1) & 1;
        const int key0 = (j_first + jj) * kBlockN;
        if (jj >= C::kStages) ok = mbar_wait(bar(C::kBarKEmpty + s), ph, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::kBarKFull + s), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(base + C::kKOff + s * C::kTileBytes + c * C::kChunkBytes, &tmK,
                      bar(C::kBarKFull + s), c * 64, key0, bh);
#ifdef FA_TEST_SKIP_ARRIVE
        // Test-only build (never in libfa.so): the stream's last V tile is
        // never loaded, so the MMA thread's bounded wait for it runs out and
        // the CTA winds down through the abort path.
        if (jj == n_stream - 1) {
          issued = 2 * jj + 1;
          break;
        }
#endif
        if (jj >= C::kStages) ok = mbar_wait(bar(C::kBarVEmpty + s), ph, abort_flag);
        if (!ok) {
          issued = 2 * jj + 1;
          break;
        }
        mbar_arrive_expect_tx(bar(C::kBarVFull + s), C::kVTileBytes);
        for (int c = 0; c < C::kChunksV; ++c)
          tma_load_3d(base + C::kVOff + s * C::kVTileBytes + c * C::kChunkBytes, &tmV,
                      bar(C::kBarVFull + s), c * 64, key0, bh);
        issued = 2 * jj + 2;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // the whole warp runs the issue loop (one elected lane issues)
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(kBlockM, DV, false, true);
      bool ok = n_stream > 0 ? mbar_wait_w(bar(C::kBarQFull), 0, abort_flag) : false;
      tc_fence_after();
      int k_ready = -1;
      auto ensure_k = [&](int jj) {
        if (ok && jj > k_ready) {
          ok = mbar_wait_w(bar(C::kBarKFull + jj % C::kStages), (jj / C::kStages) & 1, abort_flag);
          tc_fence_after();
          k_ready = jj;
        }
      };
      // Shared-memory descriptors, built once: advancing an operand by b
      // bytes adds b / 16 to the start-address field (no carry below
      // 256 KiB). The MMA thread shares its scheduler with busy softmax
      // warps, so every instruction it saves between MMAs counts.
      const uint64_t dQ0 = sdesc_sw128(base + C::kQOff, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(base + C::kKOff, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(base + C::kVOff, C::kChunkBytes, 1024);
      // S_t = Q_t K^T for stream step jj
      auto issue_s = [&](int t, int jj) {
        const uint64_t q = dQ0 + static_cast<uint64_t>(t * C::kTileBytes >> 4);
        const uint64_t k = dK0 + static_cast<uint64_t>((jj % C::kStages) * (C::kTileBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4);
          mma_ss_w(tmem + t * 128, q + off, k + off, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar(C::kBarSFull + t));
      };
      // O_t (+)= P_t V for stream step jj; P_t from its TMEM columns
      auto issue_pv = [&](int t, int jj, bool first) {
        const uint64_t v = dV0 + static_cast<uint64_t>((jj % C::kStages) * (C::kVTileBytes >> 4));
        const uint32_t pcol = C::kSepP ? C::kColP + t * 64 : t * 128;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts_w(tmem + C::kColO + t * DV, tmem + pcol + kk * 8, v + 128 * kk, kIdO,
                 (!first || kk > 0) ? 1u : 0u);
      };
      auto step_of = [&](int t, int jj) -> int {  // tile-local step, or -1
        const int a = t == 0 ? a0 : a1, b = t == 0 ? b0 : b1;
        return (jj >= a && jj < b) ? jj - a : -1;
      };
      ensure_k(0);
      if (ok) {
#pragma unroll
        for (int t = 0; t < kQTiles; ++t)
          if (step_of(t, 0) == 0) issue_s(t, 0);
        mma_commit_w(bar(C::kBarKEmpty + 0));
      }
      // The MMA thread shares its scheduler with busy softmax warps and the
      // tensor core's issue queue is short, so its loop is kept lean: when
      // both query tiles start at stream step 0 (no window) a tile's step is
      // the stream step itself.
      const bool aligned = (a0 == 0 && a1 == 0);
      if constexpr (C::kSepP) {
        if (aligned) {
          for (int jj = 0; jj < n_stream && ok; ++jj) {
#pragma unroll
            for (int t = 0; t < kQTiles; ++t) {
              if (!ok || jj + 1 >= (t == 0 ? b0 : b1)) continue;
              ok = mbar_wait_w(bar(C::kBarSFree + t), jj & 1, abort_flag);
              if (!ok) break;
              ensure_k(jj + 1);
              if (!ok) break;
              tc_fence_after();
              issue_s(t, jj + 1);
            }
            if (!ok) break;
            if (jj + 1 < n_stream) mma_commit_w(bar(C::kBarKEmpty + (jj + 1) % C::kStages));
            ok = mbar_wait_w(bar(C::kBarVFull + jj % C::kStages), (jj / C::kStages) & 1, abort_flag);
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < kQTiles; ++t) {
              if (!ok || jj >= (t == 0 ? b0 : b1)) continue;
              ok = mbar_wait_w(bar(C::kBarPFull + t), jj & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, jj, jj == 0);
              mma_commit_w(bar(C::kBarPVDone + t));
            }
            if (!ok) break;
            mma_commit_w(bar(C::kBarVEmpty + jj % C::kStages));
          }
        }
        // General case: per stream step jj, QK^T of step jj+1 for each query
        // tile as soon as its softmax holds S of step jj in registers, then
        // P.V of step jj once P is written.
        for (int jj = 0; jj < n_stream && ok && !aligned; ++jj) {
#pragma unroll
          for (int t = 0; t < kQTiles; ++t) {
            const int u = step_of(t, jj + 1);
            if (!ok || u < 0) continue;
            if (u > 0) ok = mbar_wait_w(bar(C::kBarSFree + t), (u - 1) & 1, abort_flag);
            if (!ok) break;
            ensure_k(jj + 1);
            if (!ok) break;
            tc_fence_after();
            issue_s(t, jj + 1);
          }
          if (!ok) break;
          if (jj + 1 < n_stream) mma_commit_w(bar(C::kBarKEmpty + (jj + 1) % C::kStages));
          ok = mbar_wait_w(bar(C::kBarVFull + jj % C::kStages), (jj / C::kStages) & 1, abort_flag);
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < kQTiles; ++t) {
            const int u = step_of(t, jj);
            if (!ok || u < 0) continue;
            ok = mbar_wait_w(bar(C::kBarPFull + t), u & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, jj, u == 0);
            mma_commit_w(bar(C::kBarPVDone + t));
          }
          if (!ok) break;
          mma_commit_w(bar(C::kBarVEmpty + jj % C::kStages));
        }
      } else {
        // P overwrites S: each tile's next QK^T is issued after its P.V, so
        // the P.V reads P before the new S lands in the same columns.
        if (aligned) {
          for (int jj = 0; jj < n_stream && ok; ++jj) {
            ok = mbar_wait_w(bar(C::kBarVFull + jj % C::kStages), (jj / C::kStages) & 1, abort_flag);
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < kQTiles; ++t) {
              const int bt = t == 0 ? b0 : b1;
              if (!ok || jj >= bt) continue;
              ok = mbar_wait_w(bar(C::kBarPFull + t), jj & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, jj, jj == 0);
              if (jj + 1 < bt) {
                ensure_k(jj + 1);
                if (!ok) break;
                issue_s(t, jj + 1);
              } else {
                mma_commit_w(bar(C::kBarOFinal + t));
              }
            }
            if (!ok) break;
            mma_commit_w(bar(C::kBarVEmpty + jj % C::kStages));
            if (jj + 1 < n_stream) mma_commit_w(bar(C::kBarKEmpty + (jj + 1) % C::kStages));
          }
        }
        for (int jj = 0; jj < n_stream && ok && !aligned; ++jj) {
          ok = mbar_wait_w(bar(C::kBarVFull + jj % C::kStages), (jj / C::kStages) & 1, abort_flag);
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < kQTiles; ++t) {
            const int u = step_of(t, jj);
            if (!ok || u < 0) continue;
            ok = mbar_wait_w(bar(C::kBarPFull + t), u & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, jj, u == 0);
            if (jj + 1 < (t == 0 ? b0 : b1)) {
              ensure_k(jj + 1);
              if (!ok) break;
              issue_s(t, jj + 1);
            } else {
              mma_commit_w(bar(C::kBarOFinal + t));
            }
          }
          if (!ok) break;
#pragma unroll
          for (int t = 0; t < kQTiles; ++t) {  // a tile whose range starts at step jj+1
            if (!ok || step_of(t, jj + 1) != 0) continue;
            ensure_k(jj + 1);
            if (!ok) break;
            issue_s(t, jj + 1);
          }
          if (!ok) break;
          mma_commit_w(bar(C::kBarVEmpty + jj % C::kStages));
          if (jj + 1 < n_stream) mma_commit_w(bar(C::kBarKEmpty + (jj + 1) % C::kStages));
        }
      }
      // Let every MMA this warp issued finish before TMEM is released.
      mma_commit_w(bar(C::kBarDrain));
      mbar_wait_w(bar(C::kBarDrain), 0, nullptr);
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ softmax
    const int t = warp / 4;
    const int n_mine = t == 0 ? n_t[0] : n_t[kQTiles - 1];
    const int tile_row0 = t == 0 ? q_row0[0] : q_row0[kQTiles - 1];
    const int key_tile0 = j_first + (t == 0 ? a0 : a1);  // first key tile of this query tile
    const int row = tile_row0 + (threadIdx.x & 127);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + C::kColO + t * DV;
    const uint32_t tP = tmem + lane_base + C::kColP + t * 64;  // separate-P layout only
    const float sl2 = args.scale_log2;
    // keys visible to this row: pos - window < key <= pos (pos = row + kv_off)
    const int pos = row + args.kv_off;
    const int key_hi = args.causal ? min(Nk, pos + 1) : Nk;          // exclusive
    const int key_lo = args.window ? pos - args.window + 1 : -(1 << 30);

    float m_ref = -INFINITY;  // log2-domain reference maximum
    float l = 0.f;
    bool ok = true;
    for (int u = 0; u < n_mine; ++u) {
      const int key0 = (key_tile0 + u) * kBlockN;
      // dropout: this row's keep bytes for the tile's first 64 keys, made
      // before the wait (the generator needs no operand)
      uint32_t kpre[16];
      if constexpr (kDrop) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t kb[4];
          keep_bytes_quad<true>(static_cast<uint32_t>(row >> 2), static_cast<uint32_t>((key0 + 16 * ch) >> 2),
                                static_cast<uint32_t>(bh), args.drop.offset, args.drop.seed_lo,
                                args.drop.seed_hi, kb);
#pragma unroll
          for (int q = 0; q < 4; ++q) kpre[4 * ch + q] = kb[q];
        }
      }
      ok = mbar_wait(bar(C::kBarSFull + t), u & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
      if constexpr (C::kSepP) {  // S is in registers: the next QK^T may overwrite it
        tc_fence_before();
        mbar_arrive_warp(bar(C::kBarSFree + t));
      }
      float x[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);

      if (args.window == 0) {
        // only the causal boundary tiles and the ragged last tile need a mask
        if ((args.causal && key0 + kBlockN - 1 > tile_row0 + args.kv_off) || key0 + kBlockN > Nk) {
          const int lim = key_hi - key0;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
      } else {
        const int lim_hi = key_hi - key0, lim_lo = key_lo - key0;
        if (lim_hi < kBlockN || lim_lo > 0) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim_hi || c < lim_lo) x[c] = -INFINITY;
        }
      }
      const float m_tile =
          max3(fmaxf(max32(x), max32(x + 32)), max32(x + 64), max32(x + 96)) * sl2;
      const bool need = m_tile > m_ref + kRescaleThreshold;
      const float m_old = m_ref;
      if (need) m_ref = m_tile;
      const float alpha = need ? ex2(m_old - m_ref) : 1.0f;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;

      // p = exp2(s * scale * log2(e) - m_ref), packed two at a time
      const float2 sl2x2 = make_float2(sl2, sl2);
      const float2 negm = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      const KeepTest kt = keep_test(args.drop.t);
      auto exp_half = [&](int h, uint32_t (&pk)[32]) {
        uint32_t kb[4];  // dropout, second half: keep bytes of this row for the current 16 keys
        [[maybe_unused]] uint32_t kbits = 0;  // keep bits (0x80 per kept byte) of the current key group
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 64 * h + 2 * c;
          if constexpr (kDrop) {
            if (h == 1 && (c & 7) == 0)
              keep_bytes_quad<true>(static_cast<uint32_t>(row >> 2), static_cast<uint32_t>((key0 + e) >> 2),
                                    static_cast<uint32_t>(bh), args.drop.offset, args.drop.seed_lo,
                                    args.drop.seed_hi, kb);
          }
          const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), sl2x2, negm);
          float2 pr = make_float2(ex2(a.x), ex2(a.y));
          if (c & 1) acc1 = __fadd2_rn(acc1, pr);
          else acc0 = __fadd2_rn(acc0, pr);
          pk[c] = pack_bf16(pr.x, pr.y);
          if constexpr (kDrop) {
            // keys e, e + 1 are bytes 2 (c & 1), 2 (c & 1) + 1 of key group e >> 2; a dropped
            // key's half of the bf16 pair is cleared (its p still counts in the row sum)
            if ((c & 1) == 0) kbits = keep_bits4(h == 0 ? kpre[c >> 1] : kb[(c >> 1) & 3], kt);
            pk[c] &= (c & 1) ? sign_bytes<0xBBAAu>(kbits) : sign_bytes<0x9988u>(kbits);
          }
        }
      };
      uint32_t pk[32];
      if constexpr (!C::kSepP) {
        // P columns [32h, 32h+32) hold scores [64h, 64h+64), over S
        exp_half(0, pk);
        tmem_st32(tS, pk);
        exp_half(1, pk);
        tmem_st32(tS + 32, pk);
      } else {
        exp_half(0, pk);
        // the previous step's P has been read and O accumulated once its P.V completed
        if (u > 0) {
          ok = mbar_wait(bar(C::kBarPVDone + t), (u - 1) & 1, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st32(tP, pk);
        exp_half(1, pk);
        tmem_st32(tP + 32, pk);
      }
      l = alpha * l + ((acc0.x + acc0.y) + (acc1.x + acc1.y));

      // Rescale the accumulator when this warp's maximum moved. O is settled:
      // with P over S, this tile's S MMA was committed after the previous
      // P.V; with separate P, the previous P.V has completed (waited above).
      if (u > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
          const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), al2);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(bar(C::kBarPFull + t));
    }
    const bool live = row < Nq;
    const size_t prow = (static_cast<size_t>(blockIdx.y) * args.BH + bh) * Nq + row;  // split launch
    if (ok && n_mine > 0) {
      if constexpr (C::kSepP)
        ok = mbar_wait(bar(C::kBarPVDone + t), (n_mine - 1) & 1, abort_flag);
      else
        ok = mbar_wait(bar(C::kBarOFinal + t), 0, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float inv_l = l > 0.f ? (kDrop ? args.drop.inv_keep : 1.0f) / l : 0.f;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float lse_row = l > 0.f ? (m_use + log2f(l)) * kLn2 : -INFINITY;
        const float2 il2 = make_float2(inv_l, inv_l);
        if (args.split_mode) {
          float* orow = args.part_o + prow * DV;
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
            if (live) {
              float4* dst = reinterpret_cast<float4*>(orow + c * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float2 v0 = __fmul2_rn(make_float2(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1])), il2);
                const float2 v1 = __fmul2_rn(make_float2(__uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3])), il2);
                dst[e] = make_float4(v0.x, v0.y, v1.x, v1.y);
              }
            }
          }
          if (live) args.part_lse[prow] = lse_row;
        } else {
          // A thread's O row is 128-byte lines of its own; written straight
          // from registers, one warp instruction would touch 32 lines. Each
          // warp instead swizzles its 32 rows, 64 columns at a time, into 4 KiB
          // of this tile's Q buffer (free: every QK^T of the tile has
          // completed) and writes them back as four whole lines per instruction.
          __nv_bfloat16* obase = args.o + static_cast<size_t>(bh) * Nq * DV;
          uint8_t* stage_blk = base_ptr + C::kQOff + t * C::kTileBytes + (warp & 3) * 4096;
          uint8_t* stage_row = stage_blk + lane * 128;
          const int row0 = row - lane;  // first row of this warp
#pragma unroll
          for (int h = 0; h < DV / 64; ++h) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + h * 64 + c * 32, o);
              tmem_ld_wait(o);
              uint32_t pko[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float2 v =
                    __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), il2);
                pko[e] = pack_bf16(v.x, v.y);
              }
              // 16-byte chunks 4c..4c+3 of row `lane`, chunk v in slot v ^ (lane & 7)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                *reinterpret_cast<uint4*>(stage_row + (((4 * c + e) ^ (lane & 7)) * 16)) =
                    make_uint4(pko[4 * e], pko[4 * e + 1], pko[4 * e + 2], pko[4 * e + 3]);
            }
            __syncwarp();
            // instruction j: lanes 8r'..8r'+7 write the eight chunks of row 4j + r'
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 4 * j + (lane >> 3), v = lane & 7;
              const uint4 val = *reinterpret_cast<const uint4*>(stage_blk + r * 128 + ((v ^ (r & 7)) * 16));
              if (row0 + r < Nq)
                *reinterpret_cast<uint4*>(obase + static_cast<size_t>(row0 + r) * DV + h * 64 + v * 8) = val;
            }
            __syncwarp();  // the block is read back before it is written again
          }
          if (live) args.lse[static_cast<size_t>(bh) * Nq + row] = lse_row;
        }
      }
    } else if (ok && n_mine == 0 && args.split_mode && live) {
      // no key of this split is visible to the tile: an empty partial state
      float4* dst = reinterpret_cast<float4*>(args.part_o + prow * DV);
#pragma unroll
      for (int e = 0; e < DV / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      args.part_lse[prow] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kLoadWarp && lane == 0 && *abort_flag) {
    // Every role has stopped, so the flag is final here. Consumers that gave
    // up no longer wait for the copies in flight: let every copy this thread
    // started land before the CTA exits (only the last 2 x stages can still
    // be pending: each earlier one was waited for before its slot was reused).
    mbar_wait(bar(C::kBarQFull), 0, nullptr);
    for (int x = issued - 1; x >= 0 && x >= issued - 2 * C::kStages; --x) {
      const int jj = x >> 1;
      const int s = jj % C::kStages;
      const int b = (x & 1) ? (C::kBarVFull + s) : (C::kBarKFull + s);
      mbar_wait(bar(b), (jj / C::kStages) & 1, nullptr);
    }
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(args.status, kStatusTimeout);
}

// Merges the fp32 partial states of a split key range ("FlashAttention --
// the same attention, made memory-aware", section 03: rescale each part by
// exp(m_part - m_new) and sum). In the saved-statistic form a part is
// (O_s, LSE_s) and the result is LSE = log sum_s exp(LSE_s),
// O = sum_s exp(LSE_s - LSE) O_s. One thread per 8 columns of a row.
template <int D>
__global__ void __launch_bounds__(256) fa_merge_splits(const float* __restrict__ part_o,
                                                       const float* __restrict__ part_lse,
                                                       __nv_bfloat16* __restrict__ o,
                                                       float* __restrict__ lse, int Nq, int BH,
                                                       int n_splits) {
  constexpr int kTpr = D / 8;
  constexpr int kRowsPerCta = 256 / kTpr;
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x * kRowsPerCta + threadIdx.x / kTpr;
  if (row >= Nq) return;
  const int c = (threadIdx.x % kTpr) * 8;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    float m = -INFINITY;
    for (int s = 0; s < n_splits; ++s)
      m = fmaxf(m, part_lse[(static_cast<size_t>(s) * BH + bh) * Nq + row]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float sum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < n_splits; ++s) {
        const size_t pr = (static_cast<size_t>(s) * BH + bh) * Nq + row;
        const float ls = part_lse[pr];
        if (ls == -INFINITY) continue;
        const float w = __expf(ls - m);
        sum += w;
        const float4 a = *reinterpret_cast<const float4*>(part_o + pr * D + c);
        const float4 b = *reinterpret_cast<const float4*>(part_o + pr * D + c + 4);
        acc[0] = fmaf(w, a.x, acc[0]); acc[1] = fmaf(w, a.y, acc[1]);
        acc[2] = fmaf(w, a.z, acc[2]); acc[3] = fmaf(w, a.w, acc[3]);
        acc[4] = fmaf(w, b.x, acc[4]); acc[5] = fmaf(w, b.y, acc[5]);
        acc[6] = fmaf(w, b.z, acc[6]); acc[7] = fmaf(w, b.w, acc[7]);
      }
    }
    const float inv = sum > 0.f ? 1.0f / sum : 0.f;
    const size_t orow = static_cast<size_t>(bh) * Nq + row;
    *reinterpret_cast<uint4*>(o + orow * D + c) =
        make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                   pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
    if (c == 0) lse[orow] = sum > 0.f ? m + logf(sum) : -INFINITY;
  }
}

// ---------------------------------------------------------------- persistent one-tile forward
// d = d_v = 64 over the whole key range: the one-tile CTA above, made
// persistent. A CTA of the one-tile form spends about five key tiles' worth of
// time outside its key loop (tensor-memory allocation, the first Q and K/V
// loads, the last P.V, the O write-back); at N = 2048, causal, a query tile
// has 8.5 key tiles on average, so that is a large share. Here two CTAs per SM
// each walk a list of query tiles (snake-dealt from the heaviest-first list),
// keeping the barriers, the K/V ring and the tensor memory across them: the
// next tile's Q is loaded into the second Q buffer while the current tile runs,
// and its first QK^T is issued as soon as the current tile's last S has been
// read, so it overlaps the current tile's last softmax, P.V and write-back.
//
// CTA (192 threads): warps 0-3 softmax (thread = row = TMEM lane), warp 4
// MMA issue and TMEM allocation, warp 5 TMA producer, which also writes each
// tile's geometry record for the softmax warps and issues the O write-back
// stores from the staging block they fill, so neither sits on the softmax
// warps' path between tiles.
// Tensor memory (256 columns): S [0,128), O [128,192), P (bf16 pairs) [192,256).
// Shared memory: two Q buffers, two K and two V stages (16 KiB each).
namespace pf {

constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kTileBytes = kBlockM * 64 * 2;  // 128 rows x 64 bf16, one 128-byte-swizzled chunk
constexpr int kStages = 2;
constexpr int kQOff = 0;                      // the q-th tile with work uses Q buffer q & 1
constexpr int kKOff = kQOff + 2 * kTileBytes;
constexpr int kVOff = kKOff + kStages * kTileBytes;
constexpr int kBarOff = kVOff + kStages * kTileBytes;
enum : int {
  kBarQFull = 0,               // two
  kBarOStaged = kBarQFull + 2,  // two: the tile's O rows are staged in its Q buffer (4 warps)
  kBarKFull = kBarOStaged + 2,
  kBarKEmpty = kBarKFull + kStages,
  kBarVFull = kBarKEmpty + kStages,
  kBarVEmpty = kBarVFull + kStages,
  kBarSFull = kBarVEmpty + kStages,
  kBarSFree,                   // S is in the softmax's registers (4 warps)
  kBarPFull,                   // P written, O rescaled (4 warps)
  kBarPVDone,
  kBarDrain,
  kNumBars
};
constexpr int kMiscOff = kBarOff + kNumBars * 8;
// two item records (int4: bh, row0, lo, n), 16-byte aligned for their vector accesses
constexpr int kRecOff = (kMiscOff + 16 + 15) & ~15;
static_assert(kRecOff % 16 == 0, "item records need 16-byte alignment");
constexpr int kSmemBytes = kRecOff + 32 + 1024;   // + slack to align the base
static_assert(2 * kSmemBytes <= 233472, "two persistent CTAs must fit on an SM");
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;

// One query tile (128 rows of one batch-head) and the key tiles it needs.
struct Item {
  int bh, row0;
  int lo;  // first key tile
  int n;   // key tiles (0: none)
};

// Item x of the heaviest-first list: x / BH counts query tiles from the last
// (the causal tile with the most keys), x % BH is the batch-head.
__device__ __forceinline__ Item item_geom(const FwdArgs& a, int x) {
  Item it;
  it.bh = x % a.BH;
  it.row0 = (a.num_pairs - 1 - x / a.BH) * kBlockM;
  const int n_kv = (a.Nk + kBlockN - 1) / kBlockN;
  int lo = 0, hi = n_kv;
  if (a.causal) {
    const int last_row = min(it.row0 + kBlockM, a.Nq) - 1;
    hi = min(hi, (last_row + a.kv_off) / kBlockN + 1);
  }
  if (a.window) {
    const int first_key = it.row0 + a.kv_off - a.window + 1;
    if (first_key > 0) lo = max(lo, first_key / kBlockN);
  }
  it.lo = lo;
  it.n = (it.row0 >= a.Nq || hi <= lo) ? 0 : hi - lo;
  return it;
}

// The k-th item of this CTA: round k deals items k*G .. k*G+G-1 to the CTAs,
// in reverse order on odd rounds, so the per-CTA totals stay balanced.
__device__ __forceinline__ bool item_of(int k, int num_items, int* x) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int v = k * G + ((k & 1) ? (G - 1 - c) : c);
  *x = v;
  return v < num_items;
}

template <bool kDrop>
__global__ void __launch_bounds__(kThreads, 2)
    fa_fwd_persist(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const FwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto bar = [&](int i) -> uint32_t { return base + kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kMiscOff + 4);
  const int num_items = args.num_pairs * args.BH;
  const int Nq = args.Nq, Nk = args.Nk;
  const int warp = warp_id();
  const int lane = lane_id();
  // producer: Q tiles and K/V copies started (K of stream step s is copy 2 s, its V 2 s + 1)
  int q_loaded = 0, kv_issued = 0;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarQFull + b), 1);
      mbar_init(bar(kBarOStaged + b), 4);
    }
    for (int st = 0; st < kStages; ++st) {
      mbar_init(bar(kBarKFull + st), 1);
      mbar_init(bar(kBarKEmpty + st), 1);
      mbar_init(bar(kBarVFull + st), 1);
      mbar_init(bar(kBarVEmpty + st), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 4);
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarPVDone), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();
  grid_dep_launch();

  // Every role walks the same items; q counts the items with work (their Q
  // buffer is q & 1) and u the key tiles over all of them (one stream step
  // each: it drives the K/V ring and every S/P barrier phase).
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmO);
      const uint64_t once = policy_evict_first();  // a Q tile is read by one item only
      bool ok = true;
      int q = 0, u = 0;
      // write-back coordinates of the items in Q buffers 0 and 1
      int wb_row0[2] = {0, 0}, wb_bh[2] = {0, 0};
      // Item qi's O, staged by the softmax warps in its Q buffer: one TMA
      // store per warp's 32 rows (rows past Nq are clipped by the O map).
      auto store_o = [&](int qi) {
        const int bb = qi & 1;
        ok = mbar_wait(bar(kBarOStaged + bb), (qi >> 1) & 1, abort_flag);
        if (!ok) return;
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4)
          tma_store_3d(&tmO, base + kQOff + bb * kTileBytes + w4 * 4096, 0, wb_row0[bb] + 32 * w4, wb_bh[bb]);
        bulk_commit_group();
      };
      // the record of the item in Q buffer bb, read by the softmax warps once
      // the buffer's QFull phase has completed (n = 0 ends the list)
      auto put_record = [&](int bb, int bh, int row0, int lo, int n) {
        asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(base + kRecOff + 16 * bb), "r"(bh),
                     "r"(row0), "r"(lo), "r"(n)
                     : "memory");
      };
      for (int k = 0; ok; ++k) {
        int x;
        if (!item_of(k, num_items, &x)) break;
        const Item it = item_geom(args, x);
        if (it.n == 0) continue;
        const int b = q & 1;
        // Q buffer b is free once the write-back of the tile before last, staged
        // in it, has been stored and the store has read it
        if (q >= 2) {
          store_o(q - 2);
          if (!ok) break;
          bulk_wait_read<0>();
        }
        wb_row0[b] = it.row0;
        wb_bh[b] = it.bh;
        put_record(b, it.bh, it.row0, it.lo, it.n);
        mbar_arrive_expect_tx(bar(kBarQFull + b), kTileBytes);
        tma_load_3d_hint(base + kQOff + b * kTileBytes, &tmQ, bar(kBarQFull + b), 0, it.row0, it.bh, once);
        q_loaded = ++q;
        for (int jj = 0; jj < it.n && ok; ++jj) {
          const int st = u % kStages;
          const uint32_t ph = ((u / kStages) + 1) & 1;
          const int key0 = (it.lo + jj) * kBlockN;
          if (u >= kStages) ok = mbar_wait(bar(kBarKEmpty + st), ph, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kBarKFull + st), kTileBytes);
          tma_load_3d(base + kKOff + st * kTileBytes, &tmK, bar(kBarKFull + st), 0, key0, it.bh);
          kv_issued = 2 * u + 1;
#ifdef FA_TEST_SKIP_ARRIVE
          // Test-only build (never in libfa.so): the first item's last V tile is
          // never loaded and nothing more is, so the MMA thread's bounded wait
          // for it runs out and the CTA winds down through the abort path.
          if (jj == it.n - 1) {
            ok = false;
            break;
          }
#endif
          if (u >= kStages) ok = mbar_wait(bar(kBarVEmpty + st), ph, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kBarVFull + st), kTileBytes);
          tma_load_3d(base + kVOff + st * kTileBytes, &tmV, bar(kBarVFull + st), 0, key0, it.bh);
          kv_issued = 2 * u + 2;
          ++u;
        }
      }
      if (ok) {
        // the end of the item list for the softmax warps (a plain arrival
        // completes the QFull phase they wait for), then the last two
        // write-backs
        put_record(q & 1, 0, 0, 0, 0);
        mbar_arrive(bar(kBarQFull + (q & 1)));
        for (int qi = q >= 2 ? q - 2 : 0; qi < q && ok; ++qi) store_o(qi);
      }
      bulk_wait<0>();  // the write-backs' global writes complete before the CTA exits
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // the whole warp runs the issue loop (one elected lane issues)
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(kBlockM, 64, false, true);
      // descriptors built once, advanced by byte offsets / 16
      const uint64_t dQ0 = sdesc_sw128(base + kQOff, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(base + kKOff, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(base + kVOff, kTileBytes, 1024);
      // S = Q K^T for stream step u, Q from buffer b
      auto issue_s = [&](int b, int u) {
        const uint64_t qd = dQ0 + static_cast<uint64_t>((b * kTileBytes) >> 4);
        const uint64_t kd = dK0 + static_cast<uint64_t>(((u % kStages) * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ss_w(tmem + kColS, qd + 2 * kk, kd + 2 * kk, kIdS, kk > 0 ? 1u : 0u);
        mma_commit_w(bar(kBarSFull));
      };
      // O (+)= P V for stream step u, P from its TMEM columns
      auto issue_pv = [&](int u, bool first) {
        const uint64_t vd = dV0 + static_cast<uint64_t>(((u % kStages) * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts_w(tmem + kColO, tmem + kColP + kk * 8, vd + 128 * kk, kIdO, (!first || kk > 0) ? 1u : 0u);
      };
      int k_next = 0;
      auto next_item = [&](Item* it) -> bool {  // this CTA's next item with work
        int x;
        while (item_of(k_next, num_items, &x)) {
          ++k_next;
          *it = item_geom(args, x);
          if (it->n > 0) return true;
        }
        return false;
      };
      bool ok = true;
      Item cur;
      bool have = next_item(&cur);
      int q = 0, u0 = 0;  // q: ordinal of cur among items with work; u0: stream step of its first tile
      if (have) {
        ok = mbar_wait_w(bar(kBarQFull + 0), 0, abort_flag);
        if (ok) ok = mbar_wait_w(bar(kBarKFull + 0), 0, abort_flag);
        tc_fence_after();
        if (ok) {
          issue_s(0, 0);
          mma_commit_w(bar(kBarKEmpty + 0));
        }
      }
      while (have && ok) {
        Item nxt;
        const bool have_next = next_item(&nxt);
        // S(u + 1) once the softmax holds S(u) in registers; qb: its Q buffer
        auto next_s = [&](int u, int qb, bool new_item) {
          ok = mbar_wait_w(bar(kBarSFree), u & 1, abort_flag);
          if (ok && new_item) ok = mbar_wait_w(bar(kBarQFull + qb), ((q + 1) >> 1) & 1, abort_flag);
          if (ok) ok = mbar_wait_w(bar(kBarKFull + (u + 1) % kStages), ((u + 1) / kStages) & 1, abort_flag);
          if (!ok) return;
          tc_fence_after();
          issue_s(qb, u + 1);
          mma_commit_w(bar(kBarKEmpty + (u + 1) % kStages));
        };
        for (int jj = 0; jj < cur.n && ok; ++jj) {
          const int u = u0 + jj;
          const bool last = jj + 1 == cur.n;
          // within an item: the next tile's S first, so that it computes while
          // the softmax forms P(u)
          if (!last) next_s(u, q & 1, false);
          if (!ok) break;
          ok = mbar_wait_w(bar(kBarVFull + u % kStages), (u / kStages) & 1, abort_flag);
          if (!ok) break;
          ok = mbar_wait_w(bar(kBarPFull), u & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_pv(u, jj == 0);
          mma_commit_w(bar(kBarPVDone));
          mma_commit_w(bar(kBarVEmpty + u % kStages));
          // the item's last tile: its P.V goes first, so the write-back is not held
          // up by the next item's Q and K loads; the next item's first S then
          // computes during the write-back
          if (last && have_next) next_s(u, (q + 1) & 1, true);
        }
        u0 += cur.n;
        ++q;
        cur = nxt;
        have = have_next;
      }
      // Let every MMA this warp issued finish before TMEM is released.
      mma_commit_w(bar(kBarDrain));
      mbar_wait_w(bar(kBarDrain), 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tO = tmem + lane_base + kColO;
    const uint32_t tP = tmem + lane_base + kColP;
    const float sl2 = args.scale_log2;
    bool ok = true;
    int q = 0, u = 0;
    while (ok) {
      const int b = q & 1;
      // the item's record (written by the producer before its Q load) and Q
      // tile have arrived; n = 0 ends the list
      ok = mbar_wait(bar(kBarQFull + b), (q >> 1) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int4 rec = *reinterpret_cast<const int4*>(base_ptr + kRecOff + 16 * b);
      if (rec.w == 0) break;
      Item it;
      it.bh = rec.x;
      it.row0 = rec.y;
      it.lo = rec.z;
      it.n = rec.w;
      const int bh = it.bh;
      const int row = it.row0 + (threadIdx.x & 127);
      // keys visible to this row: pos - window < key <= pos (pos = row + kv_off)
      const int pos = row + args.kv_off;
      const int key_hi = args.causal ? min(Nk, pos + 1) : Nk;  // exclusive
      const int key_lo = args.window ? pos - args.window + 1 : -(1 << 30);
      float m_ref = -INFINITY;  // log2-domain reference maximum
      float l = 0.f;
      for (int jj = 0; jj < it.n; ++jj, ++u) {
        const int key0 = (it.lo + jj) * kBlockN;
        // dropout: this row's keep bytes for the tile's first 64 keys, made
        // before the wait (the generator needs no operand)
        uint32_t kpre[16];
        if constexpr (kDrop) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t kb[4];
            keep_bytes_quad<true>(static_cast<uint32_t>(row >> 2), static_cast<uint32_t>((key0 + 16 * ch) >> 2),
                                  static_cast<uint32_t>(bh), args.drop.offset, args.drop.seed_lo,
                                  args.drop.seed_hi, kb);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) kpre[4 * ch + qq] = kb[qq];
          }
        }
        ok = mbar_wait(bar(kBarSFull), u & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
        // S is in registers: the next QK^T may overwrite it
        tc_fence_before();
        mbar_arrive_warp(bar(kBarSFree));
        float x[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
        if (args.window == 0) {
          // only the causal boundary tiles and the ragged last tile need a mask
          if ((args.causal && key0 + kBlockN - 1 > it.row0 + args.kv_off) || key0 + kBlockN > Nk) {
            const int lim = key_hi - key0;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim) x[c] = -INFINITY;
          }
        } else {
          const int lim_hi = key_hi - key0, lim_lo = key_lo - key0;
          if (lim_hi < kBlockN || lim_lo > 0) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim_hi || c < lim_lo) x[c] = -INFINITY;
          }
        }
        const float m_tile =
            max3(fmaxf(max32(x), max32(x + 32)), max32(x + 64), max32(x + 96)) * sl2;
        const bool need = m_tile > m_ref + kRescaleThreshold;
        const float m_old = m_ref;
        if (need) m_ref = m_tile;
        const float alpha = need ? ex2(m_old - m_ref) : 1.0f;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // p = exp2(s * scale * log2(e) - m_ref), packed two at a time
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 negm = make_float2(-m_use, -m_use);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        const KeepTest kt = keep_test(args.drop.t);
        auto exp_half = [&](int h, uint32_t (&pk)[32]) {
          uint32_t kb[4];  // dropout, second half: keep bytes of this row for the current 16 keys
          [[maybe_unused]] uint32_t kbits = 0;  // keep bits (0x80 per kept byte) of the current key group
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e = 64 * h + 2 * c;
            if constexpr (kDrop) {
              if (h == 1 && (c & 7) == 0)
                keep_bytes_quad<true>(static_cast<uint32_t>(row >> 2), static_cast<uint32_t>((key0 + e) >> 2),
                                      static_cast<uint32_t>(bh), args.drop.offset, args.drop.seed_lo,
                                      args.drop.seed_hi, kb);
            }
            const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), sl2x2, negm);
            float2 pr = make_float2(ex2(a.x), ex2(a.y));
            if (c & 1) acc1 = __fadd2_rn(acc1, pr);
            else acc0 = __fadd2_rn(acc0, pr);
            pk[c] = pack_bf16(pr.x, pr.y);
            if constexpr (kDrop) {
              // keys e, e + 1 are bytes 2 (c & 1), 2 (c & 1) + 1 of key group e >> 2; a dropped
              // key's half of the bf16 pair is cleared (its p still counts in the row sum)
              if ((c & 1) == 0) kbits = keep_bits4(h == 0 ? kpre[c >> 1] : kb[(c >> 1) & 3], kt);
              pk[c] &= (c & 1) ? sign_bytes<0xBBAAu>(kbits) : sign_bytes<0x9988u>(kbits);
            }
          }
        };
        uint32_t pk[32];
        exp_half(0, pk);
        // the previous step's P (this item's, or the last of the item before)
        // has been read once its P.V completed
        if (u > 0) {
          ok = mbar_wait(bar(kBarPVDone), (u - 1) & 1, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st32(tP, pk);
        exp_half(1, pk);
        tmem_st32(tP + 32, pk);
        l = alpha * l + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
        // Rescale this item's accumulator when this warp's maximum moved (its
        // previous P.V has completed: waited above).
        if (jj > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
            const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), al2);
              o[e] = __float_as_uint(v.x);
              o[e + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(kBarPFull));
      }
      if (!ok) break;
      // write-back: this item's last P.V has completed
      ok = mbar_wait(bar(kBarPVDone), (u - 1) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool live = row < Nq;
      const float inv_l = l > 0.f ? (kDrop ? args.drop.inv_keep : 1.0f) / l : 0.f;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float lse_row = l > 0.f ? (m_use + log2f(l)) * kLn2 : -INFINITY;
      const float2 il2 = make_float2(inv_l, inv_l);
      // each warp swizzles its 32 rows into 4 KiB of this item's Q buffer (every
      // QK^T of the item has completed), in the layout of the O map's 128-byte
      // swizzle; the producer stores them with TMA bulk stores (rows past Nq
      // are not written), so the warps wait neither on 32 global stores nor on
      // the store reading the block
      const int wblk = (warp & 3) * 4096;
      uint8_t* stage_blk = base_ptr + kQOff + b * kTileBytes + wblk;
      uint8_t* stage_row = stage_blk + lane * 128;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        uint32_t pko[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), il2);
          pko[e] = pack_bf16(v.x, v.y);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<uint4*>(stage_row + (((4 * c + e) ^ (lane & 7)) * 16)) =
              make_uint4(pko[4 * e], pko[4 * e + 1], pko[4 * e + 2], pko[4 * e + 3]);
      }
      fence_async_smem();  // the staged rows are visible to the producer's bulk store
      mbar_arrive_warp(bar(kBarOStaged + b));
      if (live) args.lse[static_cast<size_t>(bh) * Nq + row] = lse_row;
      ++q;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kLoadWarp && lane == 0 && *abort_flag) {
    // Every role has stopped, so the flag is final: let every copy this thread
    // started land before the CTA exits (only the last two Q tiles and the
    // last 2 x stages K/V copies can still be pending).
    for (int i = q_loaded - 1; i >= 0 && i >= q_loaded - 2; --i)
      mbar_wait(bar(kBarQFull + (i & 1)), (i >> 1) & 1, nullptr);
    for (int c = kv_issued - 1; c >= 0 && c >= kv_issued - 2 * kStages; --c) {
      const int uu = c >> 1, st = uu % kStages;
      mbar_wait(bar(((c & 1) ? kBarVFull : kBarKFull) + st), (uu / kStages) & 1, nullptr);
    }
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(args.status, kStatusTimeout);
}

}  // namespace pf

// ---------------------------------------------------------------- persistent two-tile forward
// d_v = 128 (d = 64 or 128) over the whole key range, with or without a
// window: the two-tile CTA above (P over S, O 128 columns per tile), made
// persistent. A CTA of the two-tile form spends several microseconds outside
// its key loop (tensor-memory allocation, the first Q and K/V loads with an
// empty ring, the last P.V, the O write-back) and a grid of a few waves
// leaves the last one part-empty; both weigh most on short rows (a ragged
// N = 1000 has 8 key tiles per pair, a causal pair near the diagonal or a
// window of 1024 keys a handful). Here one CTA
// per SM walks a snake-dealt share of the (pair of query tiles, batch-head)
// items, heaviest first, keeping the barriers, the K/V ring and the tensor
// memory across them: the K/V copies run on across item boundaries, the next
// item's Q is loaded as soon as the current item's last QK^T has completed,
// and its first QK^T is issued right behind the current item's last P.V, so
// it computes during the write-back. O is staged for whole-line stores in a
// block of its own, since the Q buffer holds the next item's Q by then.
//
// CTA (320 threads): warps 0-7 softmax (warpgroup t = query tile t; thread =
// row = TMEM lane), warp 8 MMA issue and TMEM allocation, warp 9 TMA producer.
// Tensor memory (512 columns): S/P of tile t [128 t, 128 t + 128), O of tile
// t [256 + 128 t, 384 + 128 t).
namespace pq {

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kChunkBytes = kBlockM * 64 * 2;  // 16 KiB: 128 rows x 64 bf16, one 128-byte-swizzled chunk
constexpr int kOStageBytes = 2 * 4 * 4096;      // 4 KiB per softmax warp

// DV = 128: S/P of tile t in [128 t, 128 t + 128) (P over S), O of tile t in
// [256 + 128 t, 384 + 128 t). DV = 64: S of tile t in [128 t, 128 t + 128), O
// in [256 + 64 t, 320 + 64 t), P in [384 + 64 t, 448 + 64 t): with P in
// columns of its own the softmax releases S as soon as it has loaded it, and
// the tile's next QK^T computes while it forms P.
template <int D, int DV>
struct Cfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunksV = DV / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;    // Q or K tile
  static constexpr int kVTileBytes = kChunksV * kChunkBytes;  // V tile
  static constexpr bool kSepP = DV == 64;
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kQOff = 0;  // tiles 0 and 1
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kOStageOff = kVOff + kStages * kVTileBytes;
  static constexpr int kBarOff = kOStageOff + kOStageBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQFree = 1;  // every QK^T of the item has completed
  static constexpr int kBarKFull = 2;
  static constexpr int kBarKEmpty = kBarKFull + kStages;
  static constexpr int kBarVFull = kBarKEmpty + kStages;
  static constexpr int kBarVEmpty = kBarVFull + kStages;
  static constexpr int kBarSFull = kBarVEmpty + kStages;  // one per tile
  static constexpr int kBarPFull = kBarSFull + 2;         // one per tile (4 warps)
  static constexpr int kBarOFinal = kBarPFull + 2;        // one per tile (P over S)
  static constexpr int kBarSFree = kBarOFinal + 2;        // one per tile (4 warps; separate P)
  static constexpr int kBarPVDone = kBarSFree + 2;        // one per tile (separate P)
  static constexpr int kBarDrain = kBarPVDone + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base
  static_assert(kSmemBytes <= 232448, "persistent two-tile forward exceeds shared memory");
  static_assert(kOStageOff % 1024 == 0, "staging blocks need 1 KiB alignment");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColP = kColO + 2 * DV;  // separate P only
  static_assert(!kSepP || kColP + 128 <= kTmemCols, "two-tile forward exceeds tensor memory");
};

// Item x of the heaviest-first list (x / BH counts query-tile pairs from the
// last, x % BH is the batch-head): its first row and the key tiles of each
// tile, [lo_t, lo_t + n_t) (the causal limit of its last row, the window's
// start for its first row; n_t = 0: the tile is past Nq). The item streams
// the union of the two ranges, key tiles [j0, j0 + ns); tile t takes part in
// stream steps [a_t, a_t + n_t), a_t = lo_t - j0.
struct Pair {
  int bh, row0;
  int n[2], a[2];
  int j0, ns;
};
__device__ __forceinline__ Pair pair_geom(const FwdArgs& a, int x) {
  Pair p;
  p.bh = x % a.BH;
  p.row0 = (a.num_pairs - 1 - x / a.BH) * 2 * kBlockM;
  const int n_kv = (a.Nk + kBlockN - 1) / kBlockN;
  int lo[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = p.row0 + t * kBlockM;
    int l = 0, hi = n_kv;
    if (a.causal) hi = min(hi, (min(r0 + kBlockM, a.Nq) - 1 + a.kv_off) / kBlockN + 1);
    if (a.window) {
      const int first_key = r0 + a.kv_off - a.window + 1;
      if (first_key > 0) l = first_key / kBlockN;
    }
    lo[t] = l;
    p.n[t] = (r0 >= a.Nq || hi <= l) ? 0 : hi - l;
  }
  // tile 1 starts no earlier than tile 0 and ends no earlier, when both have keys
  p.j0 = p.n[0] > 0 ? lo[0] : lo[1];
  const int end = max(p.n[0] > 0 ? lo[0] + p.n[0] : 0, p.n[1] > 0 ? lo[1] + p.n[1] : 0);
  p.ns = p.n[0] + p.n[1] > 0 ? end - p.j0 : 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) p.a[t] = lo[t] - p.j0;
  return p;
}

// The k-th item of this CTA: round k deals items k*G .. k*G+G-1 to the CTAs,
// in reverse order on odd rounds, so the per-CTA totals stay balanced.
__device__ __forceinline__ bool item_of(int k, int num_items, int* x) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int v = k * G + ((k & 1) ? (G - 1 - c) : c);
  *x = v;
  return v < num_items;
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_persist2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = Cfg<D, DV>;
  constexpr int kS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kMiscOff + 4);
  const int num_items = args.num_pairs * args.BH;
  const int Nq = args.Nq, Nk = args.Nk;
  const int warp = warp_id();
  const int lane = lane_id();
  // producer: Q loads and K/V copies started (K of stream step g is copy 2 g, its V 2 g + 1)
  int q_loaded = 0, kv_issued = 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQFull), 1);
    mbar_init(bar(C::kBarQFree), 1);
    for (int s = 0; s < kS; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), 4);  // one arrival per softmax warp
      mbar_init(bar(C::kBarOFinal + t), 1);
      mbar_init(bar(C::kBarSFree + t), 4);
      mbar_init(bar(C::kBarPVDone + t), 1);
    }
    mbar_init(bar(C::kBarDrain), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();
  grid_dep_launch();

  // Every role walks the same items, skipping those without work; g counts
  // stream steps (one K/V tile each) over all of them and drives the K/V
  // ring, q counts the items with work (one Q load each).
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      bool ok = true;
      int g = 0, q = 0;
      for (int k = 0; ok; ++k) {
        int x;
        if (!item_of(k, num_items, &x)) break;
        const Pair it = pair_geom(args, x);
        const int ns = it.ns;
        if (ns == 0) continue;
        for (int jj = 0; jj < ns && ok; ++jj, ++g) {
          const int st = g % kS;
          const uint32_t ph = ((g / kS) + 1) & 1;
          const int key0 = (it.j0 + jj) * kBlockN;
          if (g >= kS) ok = mbar_wait(bar(C::kBarKEmpty + st), ph, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(C::kBarKFull + st), C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(base + C::kKOff + st * C::kTileBytes + c * kChunkBytes, &tmK,
                        bar(C::kBarKFull + st), c * 64, key0, it.bh);
          kv_issued = 2 * g + 1;
          if (jj == 0) {
            // this item's Q tiles, once every QK^T of the item before has completed
            if (q > 0) ok = mbar_wait(bar(C::kBarQFree), (q - 1) & 1, abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(C::kBarQFull), (it.n[0] > 0 ? C::kTileBytes : 0) +
                                                         (it.n[1] > 0 ? C::kTileBytes : 0));
            for (int t = 0; t < 2; ++t) {
              if (it.n[t] == 0) continue;
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(base + C::kQOff + t * C::kTileBytes + c * kChunkBytes, &tmQ, bar(C::kBarQFull),
                            c * 64, it.row0 + t * kBlockM, it.bh);
            }
            q_loaded = ++q;
          }
#ifdef FA_TEST_SKIP_ARRIVE
          // Test-only build (never in libfa.so): the first item's last V tile is
          // never loaded and nothing more is, so the MMA thread's bounded wait
          // for it runs out and the CTA winds down through the abort path.
          if (jj == ns - 1) {
            ok = false;
            break;
          }
#endif
          if (g >= kS) ok = mbar_wait(bar(C::kBarVEmpty + st), ph, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(C::kBarVFull + st), C::kVTileBytes);
          for (int c = 0; c < C::kChunksV; ++c)
            tma_load_3d(base + C::kVOff + st * C::kVTileBytes + c * kChunkBytes, &tmV,
                        bar(C::kBarVFull + st), c * 64, key0, it.bh);
          kv_issued = 2 * g + 2;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // the whole warp runs the issue loop (one elected lane issues)
    constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdO = idesc_bf16_f32(kBlockM, DV, false, true);
    // descriptors built once, advanced by byte offsets / 16
    const uint64_t dQ0 = sdesc_sw128(base + C::kQOff, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(base + C::kKOff, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(base + C::kVOff, kChunkBytes, 1024);
    bool ok = true;
    int k_ready = -1;  // stream steps whose K tile is known to have landed
    auto ensure_k = [&](int gs) {
      if (ok && gs > k_ready) {
        ok = mbar_wait_w(bar(C::kBarKFull + gs % kS), (gs / kS) & 1, abort_flag);
        tc_fence_after();
        k_ready = gs;
      }
    };
    // S_t = Q_t K^T for stream step gs, into tile t's S/P columns
    auto issue_s = [&](int t, int gs) {
      const uint64_t qd = dQ0 + static_cast<uint64_t>((t * C::kTileBytes) >> 4);
      const uint64_t kd = dK0 + static_cast<uint64_t>(((gs % kS) * C::kTileBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
        mma_ss_w(tmem + t * 128, qd + off, kd + off, kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(bar(C::kBarSFull + t));
    };
    // O_t (+)= P_t V for stream step gs; P_t (bf16 pairs, 64 columns) over
    // S_t or in its own columns
    auto issue_pv = [&](int t, int gs, bool first) {
      const uint64_t vd = dV0 + static_cast<uint64_t>(((gs % kS) * C::kVTileBytes) >> 4);
      const uint32_t pcol = C::kSepP ? C::kColP + t * 64 : t * 128;
#pragma unroll
      for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_ts_w(tmem + C::kColO + t * DV, tmem + pcol + kk * 8, vd + 128 * kk, kIdO,
                 (!first || kk > 0) ? 1u : 0u);
    };
    int g = 0, q = 0;
    int ut[2] = {0, 0};  // S tiles of tile t over all items (its S/P barrier phases)
    if constexpr (C::kSepP) {
      int s_iss[2] = {0, 0};  // S tiles issued per tile
      // S_t for stream step gs once the tile's previous S is in the softmax's registers
      auto next_s = [&](int t, int gs) {
        if (s_iss[t] > 0) ok = mbar_wait_w(bar(C::kBarSFree + t), (s_iss[t] - 1) & 1, abort_flag);
        ensure_k(gs);
        if (!ok) return;
        tc_fence_after();
        issue_s(t, gs);
        ++s_iss[t];
      };
      for (int k = 0; ok; ++k) {
        int x;
        if (!item_of(k, num_items, &x)) break;
        const Pair it = pair_geom(args, x);
        const int ns = it.ns;
        if (ns == 0) continue;
        ok = mbar_wait_w(bar(C::kBarQFull), q & 1, abort_flag);
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (ok && it.n[t] > 0 && it.a[t] == 0) next_s(t, g);
        if (!ok) break;
        mma_commit_w(bar(C::kBarKEmpty + g % kS));
        if (ns == 1) mma_commit_w(bar(C::kBarQFree));
        for (int jj = 0; jj < ns && ok; ++jj) {
          const int gs = g + jj;
          // the next step's QK^T first, so that it computes while the softmax forms P
          if (jj + 1 < ns) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int u1 = jj + 1 - it.a[t];
              if (ok && u1 >= 0 && u1 < it.n[t]) next_s(t, gs + 1);
            }
            if (!ok) break;
            // every QK^T of the item has been issued: its Q buffer is free once they complete
            if (jj == ns - 2) mma_commit_w(bar(C::kBarQFree));
            mma_commit_w(bar(C::kBarKEmpty + (gs + 1) % kS));
          }
          ok = mbar_wait_w(bar(C::kBarVFull + gs % kS), (gs / kS) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int u = jj - it.a[t];
            if (!ok || u < 0 || u >= it.n[t]) continue;
            ok = mbar_wait_w(bar(C::kBarPFull + t), ut[t] & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, gs, u == 0);
            mma_commit_w(bar(C::kBarPVDone + t));
            ++ut[t];
          }
          if (!ok) break;
          mma_commit_w(bar(C::kBarVEmpty + gs % kS));
        }
        g += ns;
        ++q;
      }
    } else {
      for (int k = 0; ok; ++k) {
        int x;
        if (!item_of(k, num_items, &x)) break;
        const Pair it = pair_geom(args, x);
        const int ns = it.ns;
        if (ns == 0) continue;
        // the item's first QK^T: issued behind the previous item's last P.V
        // (in order on the tensor core, so that P.V has read P before S lands
        // in the same columns)
        ok = mbar_wait_w(bar(C::kBarQFull), q & 1, abort_flag);
        ensure_k(g);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (it.n[t] > 0 && it.a[t] == 0) issue_s(t, g);
        mma_commit_w(bar(C::kBarKEmpty + g % kS));
        if (ns == 1) mma_commit_w(bar(C::kBarQFree));
        for (int jj = 0; jj < ns && ok; ++jj) {
          const int gs = g + jj;
          ok = mbar_wait_w(bar(C::kBarVFull + gs % kS), (gs / kS) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int u = jj - it.a[t];  // tile-local step
            if (!ok || u < 0 || u >= it.n[t]) continue;
            ok = mbar_wait_w(bar(C::kBarPFull + t), ut[t] & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, gs, u == 0);
            ++ut[t];
            if (u + 1 < it.n[t]) {
              ensure_k(gs + 1);
              if (!ok) break;
              issue_s(t, gs + 1);
            } else {
              mma_commit_w(bar(C::kBarOFinal + t));
            }
          }
          if (!ok) break;
          // a tile whose range starts at the next step (a window's later start)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok || it.n[t] == 0 || it.a[t] != jj + 1) continue;
            ensure_k(gs + 1);
            if (!ok) break;
            issue_s(t, gs + 1);
          }
          if (!ok) break;
          // every QK^T of the item has been issued: its Q buffer is free once they complete
          if (jj == ns - 2) mma_commit_w(bar(C::kBarQFree));
          mma_commit_w(bar(C::kBarVEmpty + gs % kS));
          if (jj + 1 < ns) mma_commit_w(bar(C::kBarKEmpty + (gs + 1) % kS));
        }
        g += ns;
        ++q;
      }
    }
    // Let every MMA this warp issued finish before TMEM is released.
    mma_commit_w(bar(C::kBarDrain));
    mbar_wait_w(bar(C::kBarDrain), 0, nullptr);
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp / 4;  // query tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + C::kColO + t * DV;
    const uint32_t tP = tmem + lane_base + C::kColP + t * 64;  // separate P only
    const float sl2 = args.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    // this warp's staging block: 32 rows x 64 columns of O, 128-byte rows
    uint8_t* stage_blk = base_ptr + C::kOStageOff + (warp & 7) * 4096;
    uint8_t* stage_row = stage_blk + lane * 128;
    bool ok = true;
    int ut = 0, qt = 0;  // S tiles and items of this query tile so far
    for (int k = 0; ok; ++k) {
      int x;
      if (!item_of(k, num_items, &x)) break;
      const Pair it = pair_geom(args, x);
      const int n_mine = it.n[t];
      if (n_mine == 0) continue;
      const int bh = it.bh;
      const int tile_row0 = it.row0 + t * kBlockM;
      const int row = tile_row0 + (threadIdx.x & 127);
      // keys visible to this row: pos - window < key <= pos (pos = row + kv_off)
      const int pos = row + args.kv_off;
      const int key_hi = args.causal ? min(Nk, pos + 1) : Nk;          // exclusive
      const int key_lo = args.window ? pos - args.window + 1 : -(1 << 30);
      const int key_tile0 = it.j0 + it.a[t];  // this tile's first key tile
      float m_ref = -INFINITY;  // log2-domain reference maximum
      float l = 0.f;
      for (int u = 0; u < n_mine; ++u, ++ut) {
        const int key0 = (key_tile0 + u) * kBlockN;
        ok = mbar_wait(bar(C::kBarSFull + t), ut & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
        if constexpr (C::kSepP) {  // S is in registers: the tile's next QK^T may overwrite it
          tc_fence_before();
          mbar_arrive_warp(bar(C::kBarSFree + t));
        }
        float xs[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) xs[c] = __uint_as_float(sr[c >> 5][c & 31]);
        if (args.window == 0) {
          // only the causal boundary tiles and the ragged last tile need a mask
          if ((args.causal && key0 + kBlockN - 1 > tile_row0 + args.kv_off) || key0 + kBlockN > Nk) {
            const int lim = key_hi - key0;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim) xs[c] = -INFINITY;
          }
        } else {
          const int lim_hi = key_hi - key0, lim_lo = key_lo - key0;
          if (lim_hi < kBlockN || lim_lo > 0) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim_hi || c < lim_lo) xs[c] = -INFINITY;
          }
        }
        const float m_tile = max3(fmaxf(max32(xs), max32(xs + 32)), max32(xs + 64), max32(xs + 96)) * sl2;
        const bool need = m_tile > m_ref + kRescaleThreshold;
        const float m_old = m_ref;
        if (need) m_ref = m_tile;
        const float alpha = need ? ex2(m_old - m_ref) : 1.0f;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // p = exp2(s * scale * log2(e) - m_ref), packed two at a time; P
        // columns [32 h, 32 h + 32) hold scores [64 h, 64 h + 64), over S or
        // in P's own columns once the tile's previous P.V has read them
        const float2 negm = make_float2(-m_use, -m_use);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e = 64 * h + 2 * c;
            const float2 a = __ffma2_rn(make_float2(xs[e], xs[e + 1]), sl2x2, negm);
            const float2 pr = make_float2(ex2(a.x), ex2(a.y));
            if (c & 1) acc1 = __fadd2_rn(acc1, pr);
            else acc0 = __fadd2_rn(acc0, pr);
            pk[c] = pack_bf16(pr.x, pr.y);
          }
          if constexpr (C::kSepP) {
            if (h == 0 && ut > 0) {
              ok = mbar_wait(bar(C::kBarPVDone + t), (ut - 1) & 1, abort_flag);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
              tc_fence_after();
            }
            tmem_st32(tP + 32 * h, pk);
          } else {
            tmem_st32(tS + 32 * h, pk);
          }
        }
        if (!ok) break;
        l = alpha * l + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
        // Rescale the accumulator when this warp's maximum moved. O is
        // settled: this S was committed after the tile's previous P.V (P over
        // S), or that P.V's completion was waited for above (separate P).
        if (u > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
            const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), al2);
              o[e] = __float_as_uint(v.x);
              o[e + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(C::kBarPFull + t));
      }
      if (!ok) break;
      // write-back once the item's last P.V for this tile has completed; the
      // tile's next P.V (next item) waits for this warpgroup's next P, so O is
      // read out before it is overwritten
      if constexpr (C::kSepP)
        ok = mbar_wait(bar(C::kBarPVDone + t), (ut - 1) & 1, abort_flag);
      else
        ok = mbar_wait(bar(C::kBarOFinal + t), qt & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float lse_row = l > 0.f ? (m_use + log2f(l)) * kLn2 : -INFINITY;
      const float2 il2 = make_float2(inv_l, inv_l);
      // each warp swizzles its 32 rows, 64 columns at a time, into its staging
      // block and writes them back as four whole lines per instruction
      __nv_bfloat16* obase = args.o + static_cast<size_t>(bh) * Nq * DV;
      const int wrow0 = row - lane;  // first row of this warp
#pragma unroll
      for (int h = 0; h < DV / 64; ++h) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + h * 64 + c * 32, o);
          tmem_ld_wait(o);
          uint32_t pko[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), il2);
            pko[e] = pack_bf16(v.x, v.y);
          }
          // 16-byte chunks 4c..4c+3 of row `lane`, chunk v in slot v ^ (lane & 7)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint4*>(stage_row + (((4 * c + e) ^ (lane & 7)) * 16)) =
                make_uint4(pko[4 * e], pko[4 * e + 1], pko[4 * e + 2], pko[4 * e + 3]);
        }
        __syncwarp();
        // instruction j: lanes 8r'..8r'+7 write the eight chunks of row 4j + r'
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 4 * j + (lane >> 3), v = lane & 7;
          const uint4 val = *reinterpret_cast<const uint4*>(stage_blk + r * 128 + ((v ^ (r & 7)) * 16));
          if (wrow0 + r < Nq)
            *reinterpret_cast<uint4*>(obase + static_cast<size_t>(wrow0 + r) * DV + h * 64 + v * 8) = val;
        }
        __syncwarp();  // the block is read back before it is written again
      }
      if (row < Nq) args.lse[static_cast<size_t>(bh) * Nq + row] = lse_row;
      ++qt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kLoadWarp && lane == 0 && *abort_flag) {
    // Every role has stopped, so the flag is final: let every copy this thread
    // started land before the CTA exits (only the last Q load and the last
    // 2 x stages K/V copies can still be pending: each Q load waits for the
    // item before to have been consumed, and each ring slot for its last use).
    if (q_loaded > 0) mbar_wait(bar(C::kBarQFull), (q_loaded - 1) & 1, nullptr);
    for (int c = kv_issued - 1; c >= 0 && c >= kv_issued - 2 * kS; --c) {
      const int gg = c >> 1, st = gg % kS;
      mbar_wait(bar(((c & 1) ? C::kBarVFull : C::kBarKFull) + st), (gg / kS) & 1, nullptr);
    }
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(args.status, kStatusTimeout);
}

}  // namespace pq

// The persistent one-tile forward (d = d_v = 64, whole key range): at most two
// CTAs per SM, each walking its share of the query tiles.
template <bool kDrop>
int launch_fwd_persist(const FwdProblem& p, void* o, float* lse, cudaStream_t stream) {
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map_bhnd(&mq, p.q, BH, p.Nq, 64) || !make_map_bhnd(&mk, p.k, BH, p.Nk, 64) ||
      !make_map_bhnd(&mv, p.v, BH, p.Nk, 64) || !make_map_bhnd(&mo, o, BH, p.Nq, 64, 32))
    return -3;
  int* status = device_status_word();
  const int sms = device_sm_count();
  if (!status || sms <= 0) return -3;
  auto kern = pf::fa_fwd_persist<kDrop>;
  // attribute slots 15 and 16 (the other kernels use 0-14)
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), pf::kSmemBytes, kDrop ? 16 : 15)) return -3;
  FwdArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = status;
  a.Nq = p.Nq;
  a.Nk = p.Nk;
  a.kv_off = p.Nk - p.Nq;
  a.window = p.window;
  a.BH = BH;
  a.causal = p.causal ? 1 : 0;
  a.num_pairs = (p.Nq + kBlockM - 1) / kBlockM;
  a.split_tiles = (p.Nk + kBlockN - 1) / kBlockN;
  a.split_mode = 0;
  const float sl2 = p.scale * 1.4426950408889634f;
  a.scale_log2 = sl2 > 1e-30f ? sl2 : 1e-30f;
  a.drop = p.drop;
  const long long items = static_cast<long long>(a.num_pairs) * BH;
  if (items > 0x7fffffffLL) return -1;
  const long long grid = items < 2LL * sms ? items : 2LL * sms;
  const cudaError_t e = launch_overlapped(kern, dim3(static_cast<unsigned>(grid)), dim3(pf::kThreads),
                                          pf::kSmemBytes, stream, mq, mk, mv, mo, a);
  return cudaGetLastError() == cudaSuccess && e == cudaSuccess ? 0 : -3;
}

// The persistent two-tile forward (whole key range): one
// CTA per SM walks its share of the query-tile pairs.
template <int D, int DV>
int launch_fwd_persist2(const FwdProblem& p, void* o, float* lse, cudaStream_t stream) {
  using C = pq::Cfg<D, DV>;
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv;
  if (!make_map_bhnd(&mq, p.q, BH, p.Nq, D) || !make_map_bhnd(&mk, p.k, BH, p.Nk, D) ||
      !make_map_bhnd(&mv, p.v, BH, p.Nk, DV))
    return -3;
  int* status = device_status_word();
  const int sms = device_sm_count();
  if (!status || sms <= 0) return -3;
  auto kern = pq::fa_fwd_persist2<D, DV>;
  // attribute slots 17-19 (the other kernels use 0-16)
  constexpr int kSlot = DV == 64 ? 19 : (D == 128 ? 17 : 18);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes, kSlot)) return -3;
  FwdArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = status;
  a.Nq = p.Nq;
  a.Nk = p.Nk;
  a.kv_off = p.Nk - p.Nq;
  a.window = p.window;
  a.BH = BH;
  a.causal = p.causal ? 1 : 0;
  a.num_pairs = (p.Nq + 2 * kBlockM - 1) / (2 * kBlockM);
  a.split_tiles = (p.Nk + kBlockN - 1) / kBlockN;
  a.split_mode = 0;
  const float sl2 = p.scale * 1.4426950408889634f;
  a.scale_log2 = sl2 > 1e-30f ? sl2 : 1e-30f;
  a.drop = p.drop;
  const long long items = static_cast<long long>(a.num_pairs) * BH;
  if (items > 0x7fffffffLL) return -1;
  const long long grid = items < sms ? items : sms;
  const cudaError_t e = launch_overlapped(kern, dim3(static_cast<unsigned>(grid)), dim3(pq::kThreads),
                                          C::kSmemBytes, stream, mq, mk, mv, a);
  return cudaGetLastError() == cudaSuccess && e == cudaSuccess ? 0 : -3;
}

template <int D, int DV, int QT, bool kDrop = false>
int launch_fwd_d(const FwdProblem& p, void* o, float* lse, float* part_o, float* part_lse,
                 int n_splits, cudaStream_t stream) {
  using C = FwdCfg<D, DV, QT>;
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv;
  if (!make_map_bhnd(&mq, p.q, BH, p.Nq, D) || !make_map_bhnd(&mk, p.k, BH, p.Nk, D) ||
      !make_map_bhnd(&mv, p.v, BH, p.Nk, DV))
    return -3;
  int* status = device_status_word();
  if (!status) return -3;
  auto kern = fa_fwd_kernel<D, DV, QT, kDrop>;
  // attribute slots 0, 1, 4, 5, 9, 14 and with dropout 10, 11 (the backward uses 2, 3, 6-8, 12, 13)
  constexpr int kSlot = kDrop ? (QT == 1 ? 10 : 11)
                              : D == 256 ? 14 : QT == 1 ? 9 : (D == 64 ? 0 : 1) + (DV == 64 ? 0 : 4);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes, kSlot))
    return -3;
  const int n_kv = (p.Nk + kBlockN - 1) / kBlockN;
  if (n_splits < 1) n_splits = 1;
  if (n_splits > n_kv) n_splits = n_kv;
  const int split_tiles = (n_kv + n_splits - 1) / n_splits;
  n_splits = (n_kv + split_tiles - 1) / split_tiles;  // no empty trailing split
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.status = status;
  a.Nq = p.Nq;
  a.Nk = p.Nk;
  a.kv_off = p.Nk - p.Nq;
  a.window = p.window;
  a.BH = BH;
  a.causal = p.causal ? 1 : 0;
  a.num_pairs = (p.Nq + kBlockM * QT - 1) / (kBlockM * QT);
  a.split_tiles = split_tiles;
  a.split_mode = part_o != nullptr ? 1 : 0;
  // scale 0 (uniform weights) runs as a tiny positive scale: exp2 of a
  // |value| below 2^-25 rounds to exactly 1 in fp32.
  const float sl2 = p.scale * 1.4426950408889634f;
  a.scale_log2 = sl2 > 1e-30f ? sl2 : 1e-30f;
  a.drop = p.drop;
  const long long gx = static_cast<long long>(a.num_pairs) * BH;
  if (gx > 0x7fffffffLL || n_splits > 65535) return -1;
  const dim3 grid(static_cast<unsigned>(gx), a.split_mode ? n_splits : 1);
  const cudaError_t e = launch_overlapped(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, mq, mk, mv, a);
  if (cudaGetLastError() != cudaSuccess || e != cudaSuccess) return -3;
  if (a.split_mode) {
    constexpr int kRowsPerCta = 256 / (DV / 8);
    const dim3 mgrid((p.Nq + kRowsPerCta - 1) / kRowsPerCta, BH < 65535 ? BH : 65535);
    const cudaError_t em = launch_overlapped(fa_merge_splits<DV>, mgrid, dim3(256), 0, stream, part_o,
                                             part_lse, static_cast<__nv_bfloat16*>(o), lse, p.Nq, BH,
                                             n_splits);
    if (cudaGetLastError() != cudaSuccess || em != cudaSuccess) return -3;
  }
  return 0;
}

}  // namespace

int fwd_split_count(const FwdProblem& p, int n_splits, int sms) {
  const int n_kv = (p.Nk + kBlockN - 1) / kBlockN;
  if (n_splits <= 0) {
    // One CTA per SM at a time: pick the smallest split count that gives at
    // least two CTAs per SM and fills the last wave to 90 % or more (the
    // best-filled count otherwise), keeping at least four key tiles per split.
    const long long ctas = static_cast<long long>((p.Nq + 255) / 256) * p.B * p.H;
    const int s_max = n_kv / 4 > 1 ? n_kv / 4 : 1;
    int best = 1;
    double best_fill = 0.0;
    for (int s = 1; s <= s_max && s <= 256; ++s) {
      const int tiles = (n_kv + s - 1) / s, eff_s = (n_kv + tiles - 1) / tiles;
      if (eff_s != s) continue;  // would leave an empty trailing split
      const double waves = static_cast<double>(ctas * s) / sms;
      const double fill = waves / static_cast<double>(static_cast<long long>(waves + 0.999999));
      if (waves >= 2.0 && fill >= 0.9) {
        best = s;
        break;
      }
      if (fill > best_fill + 1e-9) {
        best_fill = fill;
        best = s;
      }
    }
    n_splits = best;
  }
  if (n_splits > n_kv) n_splits = n_kv;
  const int split_tiles = (n_kv + n_splits - 1) / n_splits;
  return (n_kv + split_tiles - 1) / split_tiles;
}

int launch_fwd_general(const FwdProblem& p, void* o, float* lse, float* part_o, float* part_lse,
                       int n_splits, cudaStream_t stream) {
  if (p.drop.t > 0) {  // dropout: whole key range, d = d_v in {64, 128}
    if (part_o != nullptr) return -2;
    // (the one-CTA-per-tile form: the persistent one measured no faster, 0.131 against
    // 0.130 ms on causal B=8 H=12 N=2048, p = 0.1)
    if (p.d == 64 && p.dv == 64)
      return launch_fwd_d<64, 64, 1, true>(p, o, lse, part_o, part_lse, n_splits, stream);
    if (p.d == 128 && p.dv == 128)
      return launch_fwd_d<128, 128, 2, true>(p, o, lse, part_o, part_lse, n_splits, stream);
    return -2;
  }
  if (p.d == 64 && p.dv == 64) {
    if (part_o == nullptr)  // one query tile at a time, two persistent CTAs per SM
      return launch_fwd_persist<false>(p, o, lse, stream);
    return launch_fwd_d<64, 64, 2>(p, o, lse, part_o, part_lse, n_splits, stream);
  }
  // d or d_v = 128 over the whole key range: two query tiles at a time, one
  // persistent CTA per SM (the argument checks leave no causal query before
  // the first key, which the persistent form relies on)
  const bool persist2 = part_o == nullptr && (!p.causal || p.Nk >= p.Nq);
  if (p.d == 128 && p.dv == 128) {
    if (persist2) return launch_fwd_persist2<128, 128>(p, o, lse, stream);
    return launch_fwd_d<128, 128, 2>(p, o, lse, part_o, part_lse, n_splits, stream);
  }
  // d = d_v = 256: one query tile per CTA (S 128 + O 256 tensor-memory columns)
  if (p.d == 256 && p.dv == 256) return launch_fwd_d<256, 256, 1>(p, o, lse, part_o, part_lse, n_splits, stream);
  if (p.d == 128 && p.dv == 64) {
    if (persist2) return launch_fwd_persist2<128, 64>(p, o, lse, stream);
    return launch_fwd_d<128, 64, 2>(p, o, lse, part_o, part_lse, n_splits, stream);
  }
  if (p.d == 64 && p.dv == 128) {
    if (persist2) return launch_fwd_persist2<64, 128>(p, o, lse, stream);
    return launch_fwd_d<64, 128, 2>(p, o, lse, part_o, part_lse, n_splits, stream);
  }
  return -2;
}

int launch_fwd(const Problem& p, void* o, float* lse, cudaStream_t stream) {
  FwdProblem g{p.q, p.k, p.v, p.B, p.H, p.N, p.N, p.d, p.d, p.causal, 0, p.scale, p.drop};
  return launch_fwd_general(g, o, lse, nullptr, nullptr, 1, stream);
}

}  // namespace fa
