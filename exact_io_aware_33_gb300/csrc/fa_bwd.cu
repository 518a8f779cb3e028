// Backward pass of exact attention on sm_103a, by recomputation.
//
// The forward keeps only O and the per-row log-sum-exp; the backward
// recomputes each score tile from Q and K instead of reading stored S or P
// ("FlashAttention" (Road to Intelligence), sections "The solution" and
// "What to remember"; "Flash Attention: IO-Aware Exact Attention", section
// "Storage, arithmetic and IO are separate quantities"). With
// P = exp(scale*QK^T - LSE) the gradients of L = sum(O * dO) are
//   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three kernels:
//   fa_bwd_pre   D = rowsum(dO * O) in fp32, and zero the fp32 dQ accumulator
//   fa_bwd_main  per (key/value block of 128 keys, batch-head) item: K_j and
//                V_j stay in shared memory and dK_j, dV_j accumulate in
//                tensor memory while the query blocks i stream past; per i
//                five tcgen05 MMAs:
//                  S^T  = K_j Q_i^T         (TMEM)
//                  dP^T = V_j dO_i^T        (TMEM)
//                  -> P^T, dS^T in registers (thread = key row)
//                  dV  += P^T dO_i          (P^T read from TMEM)
//                  dK  += dS^T Q_i          (dS^T read from shared memory)
//                  dQ_i = dS K_j            (same shared bytes, MN-major)
//                dQ_i is added into the fp32 accumulator in global memory.
//                Two variants: fa_bwd_main_d64 (d = d_v = 64: persistent, one
//                CTA per SM walking its share of the items, pipelined across
//                query blocks, dQ added by bulk reductions) and fa_bwd_main_seq
//                (other head sizes, one CTA per item: tensor memory too small
//                to pipeline).
//   fa_bwd_post  dQ = bf16(accumulator)
//
// The dQ accumulator is fp32 [BH, Npad, d] in a blocked layout, per group of
// 32 rows. With d = 64 (added by bulk reductions) the group is d/32 blocks of
// 32 rows x 32 columns (4 KiB, contiguous) and inside a block the eight
// 16-byte chunks of a row are rotated by XOR with (row mod 8): a block is one
// contiguous bulk reduction from a bank-conflict-free shared staging tile.
// With d = 128 (added by per-thread 16-byte reductions, thread = row) the
// group is d/4 runs of 32 rows x one 16-byte chunk, so one warp instruction
// adds 512 contiguous bytes.

#include <cuda_bf16.h>
#include <type_traits>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBlk = 128;  // keys per CTA block and queries per step
constexpr float kLog2e = 1.4426950408889634f;

struct BwdArgs {
  const float* lse2;   // [BH, Npad] -LSE * log2(e), -inf past N
  const float* Dvec;   // [BH, Npad] -rowsum(dO * O), 0 past N
  float* dq_acc;       // [BH, Npad, d] blocked layout (acc_index)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int N;
  int n_pad;
  int BH;
  int causal;
  int window;          // 0 = none; else (causal) keys j <= i - window are masked
  int n_blocks;
  float scale;
  float scale_log2;
  Dropout drop;        // kDrop kernels only (drop.inv_keep also scales dV)
};

// One past the last query block that sees a key of key block jb: with a
// window W the queries of block i reach back W - 1 positions, so only blocks
// with a query before jb*128 + 127 + W remain.
__device__ __forceinline__ int bwd_query_blocks_end(const BwdArgs& a, int jb) {
  if (!a.window) return a.n_blocks;
  const int last_query = jb * kBlk + kBlk - 1 + a.window - 1;
  const int end = last_query / kBlk + 1;
  return end < a.n_blocks ? end : a.n_blocks;
}

// Mask of the recomputed probabilities of key block jb against query block
// i, for the key at row key_row of the block: with d = query - key position,
// causal drops d < 0 and a window of W drops d >= W, i.e. the query column
// qc (within the block) is visible iff qc_lo <= qc < qc_hi. Only blocks that
// straddle a boundary (active) need the per-element test.
struct RowMask {
  int qc_lo, qc_hi;
  bool active;
};
__device__ __forceinline__ RowMask bwd_row_mask(const BwdArgs& a, int i, int jb, int key_row) {
  RowMask m;
  const int delta = (i - jb) * kBlk;  // query position minus key position at qc = key_row
  // smallest and largest d in the block: delta - 127 and delta + 127
  m.active = (a.causal && delta < kBlk - 1) || (a.window && delta + kBlk - 1 >= a.window);
  m.qc_lo = a.causal ? key_row - delta : -(1 << 30);
  m.qc_hi = a.window ? key_row - delta + a.window : (1 << 30);
  return m;
}

// Index (in floats) of dQ accumulator element (bh, row n, column c); c is
// a multiple of 4 when the caller accesses 16 bytes.
template <int D>
__host__ __device__ __forceinline__ size_t acc_index(long long bh, int n, int c, int n_pad) {
  const size_t group = (static_cast<size_t>(bh) * n_pad + (n & ~31)) * D;
  if constexpr (D == 128)
    return group + static_cast<size_t>(c >> 2) * 128 + (n & 31) * 4 + (c & 3);
  else
    return group + static_cast<size_t>(c >> 5) * 1024 + (n & 31) * 32 +
           (((((c & 31) >> 2) ^ (n & 7))) << 2) + (c & 3);
}

// ---------------------------------------------------------------- B0
// For every row of the padded [BH, Npad] grid: -D = -sum_c dO[c] * O[c] and
// -LSE * log2(e) (rows past N get 0 and -inf, so that their recomputed
// probabilities are exactly 0). Stored negated so the main kernel's packed
// FMAs take them as addends. Grid (row blocks, BH): one group of DV/8 lanes
// per row, each lane reading 8 bf16 (16 bytes) of both tensors (O and dO have
// head size DV); the CTAs of a head also zero their rows of the head's
// Npad x DQ slice of the dQ accumulator (DQ: head size of Q).
template <int DV, int DQ>
__global__ void __launch_bounds__(256) fa_bwd_pre(const __nv_bfloat16* __restrict__ o,
                                                  const __nv_bfloat16* __restrict__ dO,
                                                  const float* __restrict__ lse,
                                                  float* __restrict__ Dvec,
                                                  float* __restrict__ lse2, int N, int n_pad,
                                                  float* __restrict__ dq_acc, int BH) {
  constexpr int kTpr = DV / 8;              // lanes per row (8 or 16)
  constexpr int kRowsPerCta = 256 / kTpr;
  grid_dep_wait();
  grid_dep_launch();
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
  const int sub = threadIdx.x % kTpr;
  const int n = blockIdx.x * kRowsPerCta + threadIdx.x / kTpr;  // < n_pad (grid covers n_pad)
  const size_t head = static_cast<size_t>(bh) * N;
  const bool live = n < N;
  float acc = 0.f;
  if (live) {
    const size_t row = head + n;
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * DV + sub * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(dO + row * DV + sub * 8);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
      const float2 fb2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[e]));
      acc = fmaf(fa2.x, fb2.x, acc);
      acc = fmaf(fa2.y, fb2.y, acc);
    }
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (sub == 0 && n < n_pad) {
    const size_t prow = static_cast<size_t>(bh) * n_pad + n;
    Dvec[prow] = -acc;
    lse2[prow] = live ? -lse[head + n] * kLog2e : -INFINITY;
  }
  // zero rows [n0, n0 + kRowsPerCta) of this head's accumulator slice
  float4* z = reinterpret_cast<float4*>(dq_acc + (static_cast<size_t>(bh) * n_pad +
                                                  static_cast<size_t>(blockIdx.x) * kRowsPerCta) * DQ);
#pragma unroll
  for (int i = threadIdx.x; i < kRowsPerCta * DQ / 4; i += 256) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------- B2
// dQ = bf16(accumulator), reading the blocked accumulator layout and
// writing [BH, N, d] row-major. Grid (row blocks, BH); one thread per 8
// columns of a row (two 16-byte loads, one 16-byte store).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_post(const float* __restrict__ acc,
                                                   uint4* __restrict__ dq, int N, int n_pad, int BH) {
  constexpr int kTpr = D / 8;
  constexpr int kRowsPerCta = 256 / kTpr;
  grid_dep_wait();
  grid_dep_launch();
  const int n = blockIdx.x * kRowsPerCta + threadIdx.x / kTpr;
  if (n >= N) return;
  const int c = (threadIdx.x % kTpr) * 8;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    const float4 a = *reinterpret_cast<const float4*>(acc + acc_index<D>(bh, n, c, n_pad));
    const float4 b = *reinterpret_cast<const float4*>(acc + acc_index<D>(bh, n, c + 4, n_pad));
    dq[((static_cast<size_t>(bh) * N + n) * D + c) / 8] =
        make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
  }
}

// ---------------------------------------------------------------- B1, other head sizes
// With d = 128 (or d_v = 128) the five accumulators (S^T, dP^T, dQ, dK, dV) need 640
// tensor-memory columns of the 512, so dQ shares the dP^T columns and each
// query step runs in sequence: S^T / dP^T (one query half at a time), P/dS,
// dV / dK of the first half, dQ (as soon as both dS halves are written),
// dV / dK of the second half; dQ's read-out must finish before the next dP^T.
//
// CTA (512 threads):
//   warps 0-7  two P/dS warpgroups: thread = key row = TMEM lane; warpgroup
//              w handles query columns [64w, 64w+64) of each step, and the
//              S^T / dP^T MMAs run one query half at a time, so the first
//              half's P/dS work overlaps the second half's MMAs
//   warps 8-11 dQ warpgroup: reads dQ_i (thread = query row) and adds it
//              into global memory; writes dK, dV at the end (thread = key)
//   warp  12   tcgen05 MMA issue and TMEM allocation
//   warp  13   TMA producer; warps 14-15 idle
// TMEM columns: S^T/P^T [0,128), dP^T and dQ [128,256), dK [256,384),
// dV [384,512).
// Every wait polls (the issuing warps converged, one verdict per warp): a
// wait that sleeps in hardware wakes later than a poll notices the phase,
// and on this kernel's chain of hand-offs per step that cost more than the
// issue slots polling takes.
namespace wide {

constexpr int kHalf = 64;  // query columns per P/dS warpgroup
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kLoadWarp = 13;

// D: head size of Q and K (and of dQ, dK); DV: head size of V and dO (and dV).
template <int D, int DV>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunksV = DV / 64;
  static constexpr int kChunkBytes = kBlk * 64 * 2;
  static constexpr int kTileBytes = kChunks * kChunkBytes;    // 128 rows x d (K, Q)
  static constexpr int kVTileBytes = kChunksV * kChunkBytes;  // 128 rows x d_v (V, dO)
  static constexpr int kVecBytes = 2 * kBlk * 4;  // lse2[128], D[128] of one query block
  static constexpr int kStages = (D == 64 && DV == 64) ? 3 : 2;
  static constexpr bool kDqAliasDp = (D == 128);
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kDSOff = kVOff + kVTileBytes;            // 2 x 16 KiB
  static constexpr int kStageOff = kDSOff + 2 * kChunkBytes;
  static constexpr int kStageBytes = kTileBytes + kVTileBytes + kVecBytes;  // Q, dO, vectors
  static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = kBarQFull + kStages;
  static constexpr int kBarSFull = kBarQEmpty + kStages;    // one per query half
  static constexpr int kBarDSFull = kBarSFull + 2;           // one per query half
  static constexpr int kBarDQFull = kBarDSFull + 2;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;  // two: dQ columns [0, d/2), [d/2, d) read out
  static constexpr int kBarDKDV = kBarDQEmpty + 2;
  static constexpr int kBarDrain = kBarDKDV + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kLayoutBytes = kMiscOff + 16;
  // Slack for aligning the base to 1024 bytes, within the 227 KiB limit.
  static constexpr int kSmemLimit = 232448;
  static constexpr int kSmemBytes =
      kLayoutBytes + 1024 <= kSmemLimit ? kLayoutBytes + 1024 : kSmemLimit;
  static_assert(kLayoutBytes <= kSmemLimit, "backward tiles exceed shared memory");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDQ = kDqAliasDp ? 128 : 256;
  static constexpr uint32_t kColDK = kDqAliasDp ? 256 : 320;
  static constexpr uint32_t kColDV = kColDK + D;
  static_assert(kColDV + DV <= kTmemCols, "backward accumulators exceed tensor memory");
};

// kDrop: dropout on the probabilities (see Dropout): dV and dS use the kept
// probabilities, dS the kept and rescaled dP.
template <int D, int DV, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main_seq(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const BwdArgs args) {
  using C = BwdCfg<D, DV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kMiscOff + 4);
  if (base - raw_u32 + C::kLayoutBytes > static_cast<uint32_t>(C::kSmemBytes)) {
    // The dynamic shared memory base is not aligned enough for this layout.
    grid_dep_wait();
    if (threadIdx.x == 0) atomicExch(args.status, kStatusTimeout);
    return;
  }

  const int N = args.N;
  const int bh = blockIdx.x % args.BH;
  const int jb = static_cast<int>(blockIdx.x / args.BH);  // key block (heaviest first)
  const int i0 = args.causal ? jb : 0;
  const int n_steps = bwd_query_blocks_end(args, jb) - i0;
  const int warp = warp_id();
  const int lane = lane_id();
  int issued = 0;  // producer: query stages whose copies were started

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarQFull + s), 1);
      mbar_init(bar(C::kBarQEmpty + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kBarSFull + h), 1);
      mbar_init(bar(C::kBarDSFull + h), 4);  // one arrival per warp of warpgroup h
    }
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQEmpty), 4);
    mbar_init(bar(C::kBarDQEmpty + 1), 4);
    mbar_init(bar(C::kBarDKDV), 1);
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
      tma_prefetch_map(&tmDO);
      mbar_arrive_expect_tx(bar(C::kBarKV), C::kTileBytes + C::kVTileBytes);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(base + C::kKOff + c * C::kChunkBytes, &tmK, bar(C::kBarKV), c * 64, jb * kBlk, bh);
      for (int c = 0; c < C::kChunksV; ++c)
        tma_load_3d(base + C::kVOff + c * C::kChunkBytes, &tmV, bar(C::kBarKV), c * 64, jb * kBlk, bh);
      bool ok = true;
      for (int it = 0; it < n_steps; ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages)
          ok = mbar_wait(bar(C::kBarQEmpty + s), ((it / C::kStages) + 1) & 1, abort_flag);
        if (!ok) break;
#ifdef FA_TEST_SKIP_ARRIVE
        // Test-only build (never in libfa.so): the item's last query step is
        // never loaded, so the MMA warp's bounded wait for it runs out and the
        // CTA winds down through the abort path.
        if (it == n_steps - 1 && n_steps > 1) break;
#endif
        const int row0 = (i0 + it) * kBlk;
        const uint32_t st = base + C::kStageOff + s * C::kStageBytes;
        const uint32_t fb = bar(C::kBarQFull + s);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(st + c * C::kChunkBytes, &tmQ, fb, c * 64, row0, bh);
        for (int c = 0; c < C::kChunksV; ++c)
          tma_load_3d(st + C::kTileBytes + c * C::kChunkBytes, &tmDO, fb, c * 64, row0, bh);
        const size_t voff = static_cast<size_t>(bh) * args.n_pad + row0;
        bulk_load(st + C::kTileBytes + C::kVTileBytes, args.lse2 + voff, kBlk * 4, fb);
        bulk_load(st + C::kTileBytes + C::kVTileBytes + kBlk * 4, args.Dvec + voff, kBlk * 4, fb);
        issued = it + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // the whole warp runs the issue loop (one elected lane issues)
    {
      constexpr uint32_t kIdT = idesc_bf16_f32(kBlk, kHalf, false, false); // S^T, dP^T halves
      constexpr uint32_t kIdV = idesc_bf16_f32(kBlk, DV, false, true);     // dV
      constexpr uint32_t kIdK = idesc_bf16_f32(kBlk, D, false, true);      // dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(kBlk, D, true, true);       // dQ
      const uint32_t kb = base + C::kKOff, vb = base + C::kVOff, dsb = base + C::kDSOff;
      bool ok = mbar_wait_w(bar(C::kBarKV), 0, abort_flag);
      tc_fence_after();
      for (int it = 0; it < n_steps && ok; ++it) {
        const int s = it % C::kStages;
        ok = mbar_wait_w(bar(C::kBarQFull + s), (it / C::kStages) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qb = base + C::kStageOff + s * C::kStageBytes;
        const uint32_t dob = qb + C::kTileBytes;
        // S^T and dP^T one query half (64 columns) at a time, so the first
        // half's P/dS work overlaps the second half's MMAs
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {  // S^T_h = K Q_h^T
            const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            mma_ss_w(tmem + C::kColS + kHalf * h, sdesc_sw128(kb + off, 16, 1024),
                   sdesc_sw128(qb + off + h * 8192, 16, 1024), kIdT, kk > 0 ? 1u : 0u);
          }
          if (C::kDqAliasDp && it > 0) {  // dQ of the last step shares dP's columns, half by half
            ok = mbar_wait_w(bar(C::kBarDQEmpty + h), (it - 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk) {  // dP^T_h = V dO_h^T
            const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            mma_ss_w(tmem + C::kColDP + kHalf * h, sdesc_sw128(vb + off, 16, 1024),
                   sdesc_sw128(dob + off + h * 8192, 16, 1024), kIdT, kk > 0 ? 1u : 0u);
          }
          mma_commit_w(bar(C::kBarSFull + h));
        }
        if (!ok) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          ok = mbar_wait_w(bar(C::kBarDSFull + h), it & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          if (h == 1) {
            // dQ as soon as both dS halves are written: its read-out gates the
            // next step (dQ shares the dP^T columns at d = 128)
            if (!C::kDqAliasDp && it > 0) {
              ok = mbar_wait_w(bar(C::kBarDQEmpty + 1), (it - 1) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
            }
            // dQ = dS K          (A = dS MN-major in smem, B = K MN-major)
#pragma unroll
            for (int kk = 0; kk < kBlk / 16; ++kk)
              mma_ss_w(tmem + C::kColDQ, sdesc_sw128(dsb + kk * 2048, C::kChunkBytes, 1024),
                     sdesc_sw128(kb + kk * 2048, C::kChunkBytes, 1024), kIdQ, kk > 0 ? 1u : 0u);
            mma_commit_w(bar(C::kBarDQFull));
          }
          // dV += P_h^T dO_h   (A = P^T in TMEM, B = dO rows of half h, MN-major)
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            mma_ts_w(tmem + C::kColDV, tmem + C::kColS + kHalf * h + kk * 8,
                   sdesc_sw128(dob + (4 * h + kk) * 2048, C::kChunkBytes, 1024), kIdV,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
          // dK += dS_h^T Q_h   (A = dS^T K-major in smem region h, B = Q MN-major)
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            mma_ss_w(tmem + C::kColDK, sdesc_sw128(dsb + h * C::kChunkBytes + kk * 32, 16, 1024),
                   sdesc_sw128(qb + (4 * h + kk) * 2048, C::kChunkBytes, 1024), kIdK,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit_w(bar(C::kBarQEmpty + s));
      }
      if (ok) mma_commit_w(bar(C::kBarDKDV));
      mma_commit_w(bar(C::kBarDrain));
      mbar_wait_sleep_w(bar(C::kBarDrain), 0, nullptr);
    }
  } else if (warp < kDqWarp0) {
    // ------------------------------------------------------------ P and dS
    // warpgroup w owns query columns [64w, 64w+64) of every step
    const int w = warp >> 2;
    const int key_row = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kColS + kHalf * w;
    const uint32_t tDP = tmem + lane_base + C::kColDP + kHalf * w;
    const float sl2 = args.scale_log2;
    uint8_t* ds_base = base_ptr + C::kDSOff + w * C::kChunkBytes + key_row * 128;
    const int key_sw = key_row & 7;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const KeepTest kt = keep_test(args.drop.t);
    bool ok = true;
    for (int it = 0; it < n_steps; ++it) {
      const float* nlse2_s =
          reinterpret_cast<const float*>(base_ptr + C::kStageOff + (it % C::kStages) * C::kStageBytes +
                                         C::kTileBytes + C::kVTileBytes) + kHalf * w;
      const float* nd_s = nlse2_s + kBlk;
      // dropout: this key's keep bytes for the step's 64 query columns, made
      // before the waits (the generator needs no operand)
      uint32_t kball[16];
      if constexpr (kDrop) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t kb[4];
          keep_bytes_quad<false>(static_cast<uint32_t>((jb * kBlk + key_row) >> 2),
                                 static_cast<uint32_t>(((i0 + it) * kBlk + kHalf * w + 16 * ch) >> 2),
                                 static_cast<uint32_t>(bh), args.drop.offset, args.drop.seed_lo,
                                 args.drop.seed_hi, kb);
#pragma unroll
          for (int q = 0; q < 4; ++q) kball[4 * ch + q] = kb[q];
        }
      }
      // the stage's vectors arrive with its Q/dO tiles; S^T, dP^T with the MMA commit
      ok = mbar_wait(bar(C::kBarQFull + it % C::kStages), (it / C::kStages) & 1, abort_flag);
      if (ok) ok = mbar_wait(bar(C::kBarSFull + w), it & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const RowMask rm = bwd_row_mask(args, i0 + it, jb, key_row);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tS + c * 32, sr);
        tmem_ld32(tDP + c * 32, dr);
        tmem_ld_wait(sr);
        tmem_ld_wait(dr);
        uint32_t pp[16], dd[16];
        [[maybe_unused]] uint32_t kbits = 0;  // dropout: keep bits (0x80 per kept byte) of the current query group
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int ql = c * 32 + e;            // query column within this half
          const int qc = kHalf * w + ql;        // ... within the block
          const float2 nl = *reinterpret_cast<const float2*>(nlse2_s + ql);
          const float2 nd = *reinterpret_cast<const float2*>(nd_s + ql);
          const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                      sl2x2, nl);
          float2 p = make_float2(ex2(a.x), ex2(a.y));
          if (rm.active) {  // causal diagonal or window boundary block
            if (qc < rm.qc_lo || qc >= rm.qc_hi) p.x = 0.f;
            if (qc + 1 < rm.qc_lo || qc + 1 >= rm.qc_hi) p.y = 0.f;
          }
          const float2 dpv = make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1]));
          float2 g;
          uint32_t pkd = pack_bf16(p.x, p.y);
          if constexpr (kDrop) {
            // queries e, e + 1 are bytes (e & 3), (e & 3) + 1 of group (e >> 2) & 3: a kept
            // query's dP is scaled by 1 / (1 - p), a dropped one's is 0 and its P is cleared
            if ((e & 3) == 0) kbits = keep_bits4(kball[ql >> 2], kt);
            const uint32_t ikb = __float_as_uint(args.drop.inv_keep);
            const float2 f =
                (e & 3) ? make_float2(__uint_as_float(ikb & sign_bytes<0xAAAAu>(kbits)),
                                      __uint_as_float(ikb & sign_bytes<0xBBBBu>(kbits)))
                        : make_float2(__uint_as_float(ikb & sign_bytes<0x8888u>(kbits)),
                                      __uint_as_float(ikb & sign_bytes<0x9999u>(kbits)));
            g = __fmul2_rn(p, __ffma2_rn(dpv, f, nd));
            pkd &= (e & 3) ? sign_bytes<0xBBAAu>(kbits) : sign_bytes<0x9988u>(kbits);
          } else {
            g = __fmul2_rn(p, __fadd2_rn(dpv, nd));
          }
          pp[e >> 1] = pkd;
          dd[e >> 1] = pack_bf16(g.x, g.y);
        }
        tmem_st16(tS + c * 16, pp);
        // dS^T row of this key: 32 queries -> four swizzled 16-byte chunks
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int chunk = (c * 4 + v) ^ key_sw;
          *reinterpret_cast<uint4*>(ds_base + chunk * 16) =
              make_uint4(dd[4 * v], dd[4 * v + 1], dd[4 * v + 2], dd[4 * v + 3]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      fence_async_smem();
      mbar_arrive_warp(bar(C::kBarDSFull + w));
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ dQ, dK, dV out
    const int r = threadIdx.x - 32 * kDqWarp0;  // TMEM lane: query row of dQ, key row of dK/dV
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float scale = args.scale;
    bool ok = true;
    for (int it = 0; it < n_steps; ++it) {
      ok = mbar_wait(bar(C::kBarDQFull), it & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int q = (i0 + it) * kBlk + r;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t g[32];
        tmem_ld32(tmem + lane_base + C::kColDQ + c * 32, g);
        tmem_ld_wait(g);
        if (c == D / 64 - 1 || c == D / 32 - 1) {  // half of dQ has left tensor memory
          tc_fence_before();
          mbar_arrive_warp(bar(C::kBarDQEmpty + (c == D / 32 - 1 ? 1 : 0)));
        }
        if (q < N) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            red_add_v4(args.dq_acc + acc_index<D>(bh, q, c * 32 + e, args.n_pad),
                       __uint_as_float(g[e]) * scale,
                       __uint_as_float(g[e + 1]) * scale, __uint_as_float(g[e + 2]) * scale,
                       __uint_as_float(g[e + 3]) * scale);
        }
      }
    }
    if (ok) {
      ok = mbar_wait(bar(C::kBarDKDV), 0, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      // dK (x scale) and dV (thread = key row). Each warp swizzles its 32 rows,
      // 64 columns at a time, into 4 KiB of the query stage 0 buffer (idle:
      // every MMA has completed) and writes them back four whole 128-byte
      // lines per store instruction rather than 32 partial lines.
      tc_fence_after();
      const int lw = warp & 3;
      uint8_t* stage_blk = base_ptr + C::kStageOff + lw * 4096;
      uint8_t* stage_row = stage_blk + lane * 128;
      const int key0 = jb * kBlk + lw * 32;  // this warp's first key row
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::kColDK : C::kColDV;
        const float mul = which == 0 ? scale : args.drop.inv_keep;
        const int width = which == 0 ? D : DV;
        __nv_bfloat16* out = (which == 0 ? args.dk : args.dv) + static_cast<size_t>(bh) * N * width;
        for (int h = 0; h < width / 64; ++h) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t g[32];
            tmem_ld32(tmem + lane_base + col + h * 64 + c * 32, g);
            tmem_ld_wait(g);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16(__uint_as_float(g[2 * e]) * mul, __uint_as_float(g[2 * e + 1]) * mul);
            // 16-byte chunks 4c..4c+3 of row `lane`, chunk v in slot v ^ (lane & 7)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4*>(stage_row + (((4 * c + e) ^ (lane & 7)) * 16)) =
                  make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
          __syncwarp();
          // instruction j: lanes 8r'..8r'+7 write the eight chunks of row 4j + r'
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rr = 4 * j + (lane >> 3), v = lane & 7;
            const uint4 val = *reinterpret_cast<const uint4*>(stage_blk + rr * 128 + ((v ^ (rr & 7)) * 16));
            if (key0 + rr < N)
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(key0 + rr) * width + h * 64 + v * 8) = val;
          }
          __syncwarp();  // the block is read back before it is written again
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kLoadWarp && lane == 0 && *abort_flag) {
    // Every role has stopped, so the flag is final here: let every copy this
    // thread started land before the CTA exits (consumers that gave up no
    // longer wait for them; only the last kStages stages can be pending).
    mbar_wait_sleep(bar(C::kBarKV), 0, nullptr);
    for (int it = issued - 1; it >= 0 && it >= issued - C::kStages; --it)
      mbar_wait_sleep(bar(C::kBarQFull + it % C::kStages), (it / C::kStages) & 1, nullptr);
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(args.status, kStatusTimeout);
}

}  // namespace wide

// ---------------------------------------------------------------- B1, d = 64
// Pipelined across query blocks. The P/dS warpgroups copy S^T_i and dP^T_i
// from tensor memory into registers and release them at once, so the tensor
// core computes S^T_{i+1} and dP^T_{i+1} while P_i and dS_i are formed; P^T
// has tensor-memory columns of its own. dS has one shared-memory buffer: the
// P/dS warpgroups write dS_{i+1} once the dK and dQ MMAs of step i have read
// dS_i, which still comes before the tensor core needs dS_{i+1}.
// Two threads issue tensor-core work, each waiting on one barrier per
// query block:
//   warp 14: S^T_{i+1}, dP^T_{i+1}   (once the warpgroups hold S^T_i, dP^T_i)
//   warp 12: dQ_i = dS_i K, then dV += P^T_i dO_i, dK += dS^T_i Q_i
//            (once P_i and dS_i are written and dQ_{i-1} has been read out;
//            dQ first, so that its read-out, which gates the next query
//            block's dV/dK/dQ, starts as early as possible)
// dQ_i is added to the fp32 accumulator by the dQ warpgroup through
// per-warp 4 KiB shared staging tiles and bulk reductions (full 128-byte
// lines, no per-thread atomics).
//
// Every wait costs the issuing thread a shared-memory round trip, during
// which the tensor core's short instruction queue runs dry, so each issuer
// waits on one barrier per query block and the other roles fold their
// conditions into it: the P/dS warpgroups release S^T_i only once Q_{i+1}
// and dO_{i+1} have landed, and the dQ warpgroup joins the "dS_i written"
// barrier once it has read dQ_{i-1} (and, at an item's first query block,
// the previous item's dK and dV) out of tensor memory. With the S^T/dP^T
// MMAs on a thread of their own, neither issuer's wait holds up the other's
// instructions.
//
// Persistent: one CTA per SM walks its share of the (key block, batch-head)
// items. The query ring and every barrier phase run on a step count over
// all of the CTA's items, so the next item's first query block is already
// in flight while the current one finishes. K and V have two buffers (item
// n uses buffer n & 1), so the next item's K and V load about two query
// steps before they are needed rather than after the current item's last
// MMA; the next item's first dV/dK MMAs wait only for the current item's dK
// and dV to be read out of tensor memory.
//
// CTA (512 threads):
//   warps 0-7  two P/dS warpgroups: thread = key row = TMEM lane; warpgroup
//              w handles query columns [64w, 64w+64) of every step
//   warps 8-11 dQ warpgroup: thread = query row of dQ_i; at the end writes
//              dK and dV (thread = key row)
//   warp  12   tcgen05 MMA issue (dV, dK, dQ) and TMEM allocation
//   warp  13   TMA producer
//   warp  14   tcgen05 MMA issue (S^T, dP^T); warp 15 idle
// TMEM columns: S^T [0,128), dP^T [128,256), P^T (bf16 pairs) [256,320),
// dQ [320,384), dK [384,448), dV [448,512).
namespace pipe {

constexpr int kD = 64;
constexpr int kThreads = 512;
constexpr int kPdsThreads = 256;
constexpr int kDqWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kLoadWarp = 13;
constexpr int kSWarp = 14;
// Register budgets after the split (launch: 128 per thread x 512 threads):
// the P/dS warpgroups need more than the launch allocation, and the MMA
// warp's issue loop must not spill (its queue of MMAs is short, so every
// extra instruction between issues idles the tensor core).
constexpr uint32_t kRegsPds = 168;
constexpr uint32_t kRegsDq = 88;
constexpr uint32_t kRegsMma = 88;
static_assert(kRegsPds * kPdsThreads + kRegsDq * 128 + kRegsMma * 128 <= 128 * kThreads,
              "register split exceeds the launch allocation");

constexpr int kTileBytes = kBlk * kD * 2;           // 16 KiB, one 128B-swizzled chunk
constexpr int kVecBytes = 2 * kBlk * 4;             // -lse2[128], -D[128] of a query block
constexpr int kStages = 3;
constexpr int kKVBytes = 2 * kTileBytes;            // K then V of one item
constexpr int kKOff = 0;                            // two K/V buffers
constexpr int kVOff = kKOff + kTileBytes;
constexpr int kDSOff = kKOff + 2 * kKVBytes;        // one buffer: 2 query halves x 16 KiB
constexpr int kDSBytes = 2 * kTileBytes;
constexpr int kStageOff = kDSOff + kDSBytes;
constexpr int kStageBytes = 2 * kTileBytes + kVecBytes;  // Q, dO, vectors
constexpr int kDqStageOff = kStageOff + kStages * kStageBytes;
constexpr int kDqStageBytes = 32 * 32 * 4;          // one 32 x 32 fp32 block per dQ warp
constexpr int kBarOff = kDqStageOff + 4 * kDqStageBytes;
enum : int {
  kBarKV = 0,                // two, one per K/V buffer
  kBarKVFree = kBarKV + 2,   // two: the last MMA of the buffer's item has read K and V
  kBarQFull = kBarKVFree + 2,
  kBarQEmpty = kBarQFull + kStages,
  kBarSFull = kBarQEmpty + kStages,
  kBarSFree,     // S^T, dP^T are in registers
  kBarPFree,     // the step's dV MMA has read P^T
  kBarDSFull,    // dS written; the previous step's dQ read out
  kBarPFull,     // P^T written
  kBarDSFree,    // the step's dQ and dK MMAs have read dS
  kBarDQFull,
  kBarDKDV,
  kBarDKFree,    // an item's dK read out of tensor memory (4 dQ warps)
  kBarDVFree,    // an item's dV read out (4 dQ warps)
  kBarDrain,     // two: one per issuing thread
  kNumBars = kBarDrain + 2
};
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kLayoutBytes = kMiscOff + 16;
constexpr int kSmemBytes = kLayoutBytes + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 232448, "backward tiles exceed shared memory");
static_assert(kStageBytes % 1024 == 0 && kDqStageOff % 1024 == 0, "swizzle atoms need 1 KiB alignment");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDQ = 320, kColDK = 384, kColDV = 448;

// The k-th work item of this CTA in a snake-ordered round robin over the
// items (key block jb, batch-head bh) listed heaviest first: round k hands
// item k*G + c to CTA c, reversed on odd rounds, so the per-CTA totals stay
// balanced. Returns false when the CTA has no k-th item.
__device__ __forceinline__ bool item_of(int k, int num_items, int* x) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int v = k * G + ((k & 1) ? (G - 1 - c) : c);
  *x = v;
  return v < num_items;
}

template <bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main_d64(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto bar = [&](int i) -> uint32_t { return base + kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kMiscOff + 4);

  const int num_items = args.n_blocks * args.BH;
  // geometry of item x: key block, batch-head, first query block, query steps
  auto geom = [&](int x, int& jb, int& bh, int& i0, int& n_steps) {
    jb = x / args.BH;
    bh = x - jb * args.BH;
    i0 = args.causal ? jb : 0;
    n_steps = bwd_query_blocks_end(args, jb) - i0;
  };
  const int warp = warp_id();
  const int lane = lane_id();
  // producer: query steps and K/V items whose copies were started
  int loaded_steps = 0, loaded_kv = 0;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarKV + b), 1);
      mbar_init(bar(kBarKVFree + b), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), kPdsThreads / 32);  // one arrival per warp
    mbar_init(bar(kBarPFree), 1);
    mbar_init(bar(kBarDSFull), kPdsThreads / 32 + 4);  // one arrival per warp
    mbar_init(bar(kBarPFull), kPdsThreads / 32);
    mbar_init(bar(kBarDSFree), 1);
    mbar_init(bar(kBarDQFull), 1);
    mbar_init(bar(kBarDKDV), 1);
    mbar_init(bar(kBarDKFree), 4);
    mbar_init(bar(kBarDVFree), 4);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrain + 1), 1);
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
  if (warp >= kMmaWarp) regs_decrease<kRegsMma>();
  else if (warp >= kDqWarp0) regs_decrease<kRegsDq>();

  // Every role walks the same item sequence; g counts this CTA's query
  // steps over all its items and drives every ring slot and barrier phase.
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmDO);
      int& g = loaded_steps;
      int& n_kv = loaded_kv;
      bool ok = true;
      auto load_q = [&](int bh, int row0) {  // query block of global step g
        const int s = g % kStages;
        if (g >= kStages) ok = mbar_wait(bar(kBarQEmpty + s), ((g / kStages) + 1) & 1, abort_flag);
        if (!ok) return;
        const uint32_t st = base + kStageOff + s * kStageBytes;
        const uint32_t fb = bar(kBarQFull + s);
        mbar_arrive_expect_tx(fb, kStageBytes);
        tma_load_3d(st, &tmQ, fb, 0, row0, bh);
        tma_load_3d(st + kTileBytes, &tmDO, fb, 0, row0, bh);
        const size_t voff = static_cast<size_t>(bh) * args.n_pad + row0;
        bulk_load(st + 2 * kTileBytes, args.lse2 + voff, kBlk * 4, fb);
        bulk_load(st + 2 * kTileBytes + kBlk * 4, args.Dvec + voff, kBlk * 4, fb);
        ++g;
      };
      for (int n = 0; ok; ++n) {
        int x, jb, bh, i0, ns;
        if (!item_of(n, num_items, &x)) break;
        geom(x, jb, bh, i0, ns);
        // the item's first query block goes into the ring before its K/V;
        // K/V buffer n & 1 is free once item n - 2's last MMA has read it
        load_q(bh, i0 * kBlk);
        if (!ok) break;
        const int kv = n & 1;
        if (n >= 2) ok = mbar_wait(bar(kBarKVFree + kv), ((n >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kBarKV + kv), 2 * kTileBytes);
        // an item's K and V are read once (evict first): the L2 keeps the Q/dO
        // blocks and dQ accumulator rows that the other items re-read
        // (301 instead of 334 MB of DRAM traffic per launch, same time)
        const uint64_t once = policy_evict_first();
        tma_load_3d_hint(base + kKOff + kv * kKVBytes, &tmK, bar(kBarKV + kv), 0, jb * kBlk, bh, once);
        tma_load_3d_hint(base + kVOff + kv * kKVBytes, &tmV, bar(kBarKV + kv), 0, jb * kBlk, bh, once);
        ++n_kv;
        for (int it = 1; it < ns && ok; ++it) {
#ifdef FA_TEST_SKIP_ARRIVE
          // Test-only build (never in libfa.so): the first item's last query
          // step is never loaded and nothing more is, so the issuing warps'
          // bounded waits for it run out and the CTA winds down.
          if (n == 0 && it == ns - 1) {
            ok = false;
            break;
          }
#endif
          load_q(bh, (i0 + it) * kBlk);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // the whole warp runs the issue loop (one elected lane issues)
    {
      constexpr uint32_t kIdKV = idesc_bf16_f32(kBlk, kD, false, true);     // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(kBlk, kD, true, true);       // dQ
      // Shared-memory descriptors, built once (K and V: once per item).
      // Advancing an operand by b bytes adds b / 16 to the descriptor's
      // start-address field, which cannot carry out of its 14 bits below
      // 256 KiB.
      const uint64_t kQmn0 = sdesc_sw128(base + kStageOff, kTileBytes, 1024);
      const uint64_t kDS0 = sdesc_sw128(base + kDSOff, 16, 1024);       // dS buffer 0, K-major
      const uint64_t kDSmn0 = sdesc_sw128(base + kDSOff, kTileBytes, 1024);
      constexpr uint64_t kStageStep = kStageBytes >> 4, kTileStep = kTileBytes >> 4;
      bool ok = true;
      int g = 0;
      for (int n = 0; ok; ++n) {
        int x, jb, bh, i0, ns;
        if (!item_of(n, num_items, &x)) break;
        geom(x, jb, bh, i0, ns);
        const int kv = n & 1;
        const uint32_t kvb = base + kv * kKVBytes;
        // K has landed: the S^T MMAs that read it completed before this
        // step's P and dS were formed
        const uint64_t kKmn = sdesc_sw128(kvb + kKOff, kTileBytes, 1024);  // K as MN-major B
        for (int it = 0; it < ns && ok; ++it, ++g) {
          // P^T and dS of step g written, dQ of step g-1 read out of tensor
          // memory (at an item's first step the previous item's dK and dV
          // read-outs are waited for separately, just before dK and dV)
          ok = mbar_wait_w(bar(kBarDSFull), g & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t qmn = kQmn0 + (g % kStages) * kStageStep, omn = qmn + kTileStep;
          const uint64_t dsk = kDS0, dsmn = kDSmn0;
          // dQ = dS K first, so the dQ warpgroup starts reading it out sooner
          // (A = dS MN-major: the same bytes as dS^T, B = K MN-major)
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk)
            mma_ss_w(tmem + kColDQ, dsmn + 128 * kk, kKmn + 128 * kk, kIdQ, kk > 0 ? 1u : 0u);
          mma_commit_w(bar(kBarDQFull));
          if (it == 0 && n > 0) {  // the previous item's dK has been read out
            ok = mbar_wait_w(bar(kBarDKFree), (n - 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
          }
          // dK += dS^T Q   (A = dS^T K-major, query halves in two 16 KiB regions; B = Q MN-major)
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk)
            mma_ss_w(tmem + kColDK, dsk + (kk >> 2) * kTileStep + (kk & 3) * 2, qmn + 128 * kk, kIdKV,
                   (it > 0 || kk > 0) ? 1u : 0u);
          // the dS buffer is free once dQ and dK have read it: the P/dS warps
          // write the next step's dS while dV runs
          mma_commit_w(bar(kBarDSFree));
          // dV += P^T dO   (A = P^T bf16 pairs in TMEM, B = dO MN-major, 16 rows per step)
          ok = mbar_wait_w(bar(kBarPFull), g & 1, abort_flag);
          if (ok && it == 0 && n > 0) ok = mbar_wait_w(bar(kBarDVFree), (n - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk)
            mma_ts_w(tmem + kColDV, tmem + kColP + kk * 8, omn + 128 * kk, kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(bar(kBarPFree));
          mma_commit_w(bar(kBarQEmpty + g % kStages));
        }
        if (!ok) break;
        mma_commit_w(bar(kBarDKDV));    // dK, dV of this item are complete
        // and this K/V buffer may be refilled (the item's S^T/dP^T MMAs on
        // the other issuer completed before its last P and dS were formed)
        mma_commit_w(bar(kBarKVFree + kv));
      }
      mma_commit_w(bar(kBarDrain));
      mbar_wait_w(bar(kBarDrain), 0, nullptr);
    }
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ S^T / dP^T issue
    // the whole warp runs the issue loop (one elected lane issues)
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBlk, kBlk, false, false);
      const uint64_t kQ0 = sdesc_sw128(base + kStageOff, 16, 1024);  // stage 0 Q, K-major
      constexpr uint64_t kStageStep = kStageBytes >> 4, kTileStep = kTileBytes >> 4;
      // S^T = K Q^T and dP^T = V dO^T of global step g (both K-major)
      auto issue_sdp = [&](int g, uint64_t kK, uint64_t kV) {
        const uint64_t q = kQ0 + (g % kStages) * kStageStep, o = q + kTileStep;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss_w(tmem + kColS, kK + 2 * kk, q + 2 * kk, kIdS, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss_w(tmem + kColDP, kV + 2 * kk, o + 2 * kk, kIdS, kk > 0 ? 1u : 0u);
        mma_commit_w(bar(kBarSFull));
      };
      bool ok = true;
      int g = 0;
      for (int n = 0; ok; ++n) {
        int x, jb, bh, i0, ns;
        if (!item_of(n, num_items, &x)) break;
        geom(x, jb, bh, i0, ns);
        const int kv = n & 1;
        const uint32_t kvb = base + kv * kKVBytes;
        const uint64_t kK = sdesc_sw128(kvb + kKOff, 16, 1024);
        const uint64_t kV = sdesc_sw128(kvb + kVOff, 16, 1024);
        ok = mbar_wait_w(bar(kBarKV + kv), (n >> 1) & 1, abort_flag);
        if (ok) ok = mbar_wait_w(bar(kBarQFull + g % kStages), (g / kStages) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        issue_sdp(g, kK, kV);
        // S^T of every step is released before the next S^T is issued (the
        // next item's first one included)
        for (int it = 0; it < ns && ok; ++it, ++g) {
          ok = mbar_wait_w(bar(kBarSFree), g & 1, abort_flag);
          if (!ok) break;
          if (it + 1 < ns) {
            // the next step's Q and dO: waited for here rather than by the P/dS
            // warps, whose step must not wait on a load it does not read
            ok = mbar_wait_w(bar(kBarQFull + (g + 1) % kStages), ((g + 1) / kStages) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_sdp(g + 1, kK, kV);
          }
        }
      }
      // Let every MMA this warp issued finish before TMEM is released.
      mma_commit_w(bar(kBarDrain + 1));
      mbar_wait_w(bar(kBarDrain + 1), 0, nullptr);
    }
  } else if (warp < kDqWarp0) {
    // ------------------------------------------------------------ P and dS
    regs_increase<kRegsPds>();
    const int w = warp >> 2;  // query columns [64w, 64w+64) of every step
    const int key_row = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 64 * w;
    const uint32_t tDP = tmem + lane_base + kColDP + 64 * w;
    const uint32_t tP = tmem + lane_base + kColP + 32 * w;
    const float sl2 = args.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const int key_sw = key_row & 7;
    const KeepTest kt = keep_test(args.drop.t);
    bool ok = true;
    int g = 0;
    for (int n = 0; ok; ++n) {
      int xi, jb, bh, i0, ns;
      if (!item_of(n, num_items, &xi)) break;
      geom(xi, jb, bh, i0, ns);
    for (int it = 0; it < ns; ++it, ++g) {
      const int s = g % kStages;
      const float* nlse2_s =
          reinterpret_cast<const float*>(base_ptr + kStageOff + s * kStageBytes + 2 * kTileBytes) + 64 * w;
      const float* nd_s = nlse2_s + kBlk;
      // dropout: this key's keep bytes for the step's 64 query columns, made
      // before the waits below (the generator needs no operand) so that they
      // cost no time on the step's chain and hold no registers next to S, dP
      uint32_t kball[16];
      if constexpr (kDrop) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t kb[4];
          keep_bytes_quad<false>(static_cast<uint32_t>((jb * kBlk + key_row) >> 2),
                                 static_cast<uint32_t>(((i0 + it) * kBlk + 64 * w + 16 * ch) >> 2),
                                 static_cast<uint32_t>(bh), args.drop.offset, args.drop.seed_lo,
                                 args.drop.seed_hi, kb);
#pragma unroll
          for (int q = 0; q < 4; ++q) kball[4 * ch + q] = kb[q];
        }
      }
      // S^T, dP^T arrive with the MMA commit; the stage's vectors with its
      // Q/dO tiles (which S^T, dP^T needed, so that wait is already satisfied
      // and only makes the vectors visible here)
      ok = mbar_wait(bar(kBarSFull), g & 1, abort_flag);
      if (ok) ok = mbar_wait(bar(kBarQFull + s), (g / kStages) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32], d0[32], d1[32];
      tmem_ld32(tS, s0);
      tmem_ld32(tS + 32, s1);
      tmem_ld32(tDP, d0);
      tmem_ld32(tDP + 32, d1);
      tmem_ld_wait(s0);
      tmem_ld_wait(s1);
      tmem_ld_wait(d0);
      tmem_ld_wait(d1);
      // S^T and dP^T of this step are in registers: the next step's MMAs may
      // overwrite their columns (its Q and dO have landed, checked above).
      tc_fence_before();
      mbar_arrive_warp(bar(kBarSFree));

      const RowMask rm = bwd_row_mask(args, i0 + it, jb, key_row);
      const bool win = args.window != 0 && rm.active;
      const bool diag = args.causal && it == 0;
      uint32_t pp[32], dd[32];
      // kind 0: no mask (the causal diagonal block is masked afterwards, on
      // the packed words); 2: window boundary block. A compile-time kind
      // keeps the unmasked blocks free of per-element tests.
      auto half = [&](auto kind, const uint32_t (&sr)[32], const uint32_t (&dr)[32], int c) {
        constexpr int kKind = decltype(kind)::value;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int ql = c * 32 + e;     // query column within this warpgroup's half
          const int qc = 64 * w + ql;    // ... within the query block
          const float4 nl = *reinterpret_cast<const float4*>(nlse2_s + ql);
          const float4 nd = *reinterpret_cast<const float4*>(nd_s + ql);
          [[maybe_unused]] uint32_t kbits = 0;  // dropout: keep bits (0x80 per kept byte) of queries ql .. ql + 3
          if constexpr (kDrop) kbits = keep_bits4(kball[ql >> 2], kt);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float2 nl2 = u ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y);
            const float2 nd2 = u ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y);
            const int x = e + 2 * u;
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[x]), __uint_as_float(sr[x + 1])),
                                        sl2x2, nl2);
            float2 p = make_float2(ex2(a.x), ex2(a.y));
            if constexpr (kKind == 2) {  // window boundary (or causal diagonal) block
              const int q0 = qc + 2 * u;
              if (q0 < rm.qc_lo || q0 >= rm.qc_hi) p.x = 0.f;
              if (q0 + 1 < rm.qc_lo || q0 + 1 >= rm.qc_hi) p.y = 0.f;
            }
            const float2 dpv = make_float2(__uint_as_float(dr[x]), __uint_as_float(dr[x + 1]));
            float2 gs;
            uint32_t pkd = pack_bf16(p.x, p.y);
            if constexpr (kDrop) {
              // queries x, x + 1 are bytes 2u, 2u + 1 of kbits: a kept query's dP is scaled by
              // 1 / (1 - p), a dropped one's is 0 and its half of the P^T pair is cleared
              const uint32_t ikb = __float_as_uint(args.drop.inv_keep);
              const float2 f =
                  u ? make_float2(__uint_as_float(ikb & sign_bytes<0xAAAAu>(kbits)),
                                  __uint_as_float(ikb & sign_bytes<0xBBBBu>(kbits)))
                    : make_float2(__uint_as_float(ikb & sign_bytes<0x8888u>(kbits)),
                                  __uint_as_float(ikb & sign_bytes<0x9999u>(kbits)));
              gs = __fmul2_rn(p, __ffma2_rn(dpv, f, nd2));
              pkd &= u ? sign_bytes<0xBBAAu>(kbits) : sign_bytes<0x9988u>(kbits);
            } else {
              gs = __fmul2_rn(p, __fadd2_rn(dpv, nd2));
            }
            pp[(ql >> 1) + u] = pkd;
            dd[(ql >> 1) + u] = pack_bf16(gs.x, gs.y);
          }
        }
      };
      if (win) {
        half(std::integral_constant<int, 2>{}, s0, d0, 0);
        half(std::integral_constant<int, 2>{}, s1, d1, 1);
      } else {
        half(std::integral_constant<int, 0>{}, s0, d0, 0);
        half(std::integral_constant<int, 0>{}, s1, d1, 1);
        if (diag) {
          // Causal diagonal block, through the unmasked code above (which is
          // hot; a masked copy of it ran cold once per item): query column
          // 64 w + j comes before this key for j < lim, and there P and dS
          // are 0, so those halves of the packed words are cleared.
          const int lim = key_row - 64 * w;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int t = lim - 2 * i;  // masked elements among 2i, 2i + 1
            const uint32_t m = t <= 0 ? 0xffffffffu : (t == 1 ? 0xffff0000u : 0u);
            pp[i] &= m;
            dd[i] &= m;
          }
        }
      }

      // dS^T row of this key into the dS buffer once step g-1's dQ and dK
      // MMAs have read it (step g-1's dV may still run): 64 queries -> eight
      // swizzled 16-byte chunks
      if (g > 0) {
        ok = mbar_wait(bar(kBarDSFree), (g - 1) & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      uint8_t* ds_row = base_ptr + kDSOff + w * kTileBytes + key_row * 128;
#pragma unroll
      for (int v = 0; v < 8; ++v)
        *reinterpret_cast<uint4*>(ds_row + ((v ^ key_sw) * 16)) =
            make_uint4(dd[4 * v], dd[4 * v + 1], dd[4 * v + 2], dd[4 * v + 3]);
      fence_async_smem();
      mbar_arrive_warp(bar(kBarDSFull));
      // P^T into its own columns once the previous step's dV MMA has read them
      if (g > 0) {
        ok = mbar_wait(bar(kBarPFree), (g - 1) & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st32(tP, pp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(bar(kBarPFull));
    }
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ dQ, dK, dV out
    const int qw = warp - kDqWarp0;  // TMEM lanes [32 qw, 32 qw + 32)
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t stage = base + kDqStageOff + qw * kDqStageBytes;
    uint8_t* stage_row = base_ptr + kDqStageOff + qw * kDqStageBytes + lane * 128;
    const float scale = args.scale;
    bool ok = true;
    bool pending = false;
    // one 32 x 32 block of dQ (this warp's rows, 32 columns) -> staging -> bulk add
    auto put_block = [&](const uint32_t (&gr)[32], float* dst) {
      if (pending) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
#pragma unroll
      for (int v = 0; v < 8; ++v)
        *reinterpret_cast<float4*>(stage_row + ((v ^ (lane & 7)) * 16)) =
            make_float4(__uint_as_float(gr[4 * v]) * scale, __uint_as_float(gr[4 * v + 1]) * scale,
                        __uint_as_float(gr[4 * v + 2]) * scale, __uint_as_float(gr[4 * v + 3]) * scale);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_reduce_add_f32(dst, stage, kDqStageBytes);
        bulk_commit_group();
      }
      pending = true;
    };
    int g = 0;
    mbar_arrive_warp(bar(kBarDSFull));  // the first step has no dQ to read out
    for (int n = 0; ok; ++n) {
      int xi, jb, bh, i0, ns;
      if (!item_of(n, num_items, &xi)) break;
      geom(xi, jb, bh, i0, ns);
      for (int it = 0; it < ns; ++it, ++g) {
        ok = mbar_wait(bar(kBarDQFull), g & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // rows [32 qw, 32 qw + 32) of query block i0 + it: two contiguous 4 KiB blocks
        float* dst = args.dq_acc + (static_cast<size_t>(bh) * args.n_pad + (i0 + it) * kBlk + 32 * qw) * kD;
        uint32_t gr[32];
        tmem_ld32(tmem + lane_base + kColDQ, gr);
        tmem_ld_wait(gr);
        put_block(gr, dst);
        tmem_ld32(tmem + lane_base + kColDQ + 32, gr);
        tmem_ld_wait(gr);
        tc_fence_before();
        mbar_arrive_warp(bar(kBarDSFull));  // dQ columns free for step g+1
        put_block(gr, dst + 1024);
      }
      if (!ok) break;
      // dK (x scale) and dV of this item's keys (thread = key row); their TMEM
      // columns go to the next item right after the last read. A thread's
      // row is one 128-byte line, so storing rows straight from registers
      // would touch 32 lines per warp instruction and crowd the shared-memory
      // data path the tensor core reads its operands through; each warp
      // instead swizzles its 32 rows into its 4 KiB staging block and writes
      // them back four whole lines per instruction.
      ok = mbar_wait(bar(kBarDKDV), n & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if (pending) {  // the last dQ reduction has finished reading the staging block
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        pending = false;
      }
      const int key0 = jb * kBlk + qw * 32;  // this warp's first key row
      const uint8_t* stage_blk = base_ptr + kDqStageOff + qw * kDqStageBytes;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? kColDK : kColDV;
        const float mul = which == 0 ? scale : args.drop.inv_keep;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t gr[32];
          tmem_ld32(tmem + lane_base + col + c * 32, gr);
          tmem_ld_wait(gr);
          if (c == kD / 32 - 1) {  // this item's dK (dV) columns free for the next item
            tc_fence_before();
            mbar_arrive_warp(bar(which == 0 ? kBarDKFree : kBarDVFree));
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(gr[2 * e]) * mul, __uint_as_float(gr[2 * e + 1]) * mul);
          // 16-byte chunks 4c..4c+3 of row `lane`, chunk v in slot v ^ (lane & 7)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint4*>(stage_row + (((4 * c + e) ^ (lane & 7)) * 16)) =
                make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
        __syncwarp();
        // instruction j: lanes 8r'..8r'+7 write the eight chunks of row 4j + r'
        __nv_bfloat16* out = (which == 0 ? args.dk : args.dv) + static_cast<size_t>(bh) * args.N * kD;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 4 * j + (lane >> 3), v = lane & 7;
          const uint4 val = *reinterpret_cast<const uint4*>(stage_blk + r * 128 + ((v ^ (r & 7)) * 16));
          if (key0 + r < args.N)
            *reinterpret_cast<uint4*>(out + static_cast<size_t>(key0 + r) * kD + v * 8) = val;
        }
        __syncwarp();  // the block is read back before it is written again
      }
    }
    // the bulk reductions complete before the CTA exits
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kLoadWarp && lane == 0 && *abort_flag) {
    // Every role has stopped, so the flag is final here: let every copy this
    // thread started land before the CTA exits (consumers that gave up no
    // longer wait for them; only the last two K/V loads and the last kStages
    // query stages can be pending).
    for (int m = loaded_kv - 1; m >= 0 && m >= loaded_kv - 2; --m)
      mbar_wait(bar(kBarKV + (m & 1)), (m >> 1) & 1, nullptr);
    for (int q = loaded_steps - 1; q >= 0 && q >= loaded_steps - kStages; --q)
      mbar_wait(bar(kBarQFull + q % kStages), (q / kStages) & 1, nullptr);
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(args.status, kStatusTimeout);
}

}  // namespace pipe

// Workspace sections: D and lse2 (fp32 [BH, Npad] each), then the fp32 dQ
// accumulator [BH, Npad, d] (blocked, acc_index). Npad * 4 bytes is a
// multiple of 512, so every section and every query block's vector slice is
// 512-byte aligned.
struct Workspace {
  float* Dvec;
  float* lse2;
  float* acc;
  int n_pad;
  long long pad_rows;
};

Workspace carve(const Problem& p, void* workspace) {
  Workspace w;
  w.n_pad = (p.N + kBlk - 1) / kBlk * kBlk;
  w.pad_rows = static_cast<long long>(p.B) * p.H * w.n_pad;
  w.Dvec = static_cast<float*>(workspace);
  w.lse2 = w.Dvec + w.pad_rows;
  w.acc = w.lse2 + w.pad_rows;
  return w;
}

template <int DV, int DQ>
int launch_pre_d(const Problem& p, const void* o, const float* lse, const void* dO,
                 void* workspace, cudaStream_t stream) {
  const Workspace w = carve(p, workspace);
  constexpr int kRowsPerCta = 256 / (DV / 8);
  const int BH = p.B * p.H;
  const dim3 grid(w.n_pad / kRowsPerCta, BH < 65535 ? BH : 65535);
  const cudaError_t e =
      launch_overlapped(fa_bwd_pre<DV, DQ>, grid, dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(o),
                        static_cast<const __nv_bfloat16*>(dO), lse, w.Dvec, w.lse2, p.N, w.n_pad, w.acc, BH);
  return cudaGetLastError() == cudaSuccess && e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

BwdArgs make_args(const Problem& p, const Workspace& w, void* dk, void* dv, int* status) {
  BwdArgs a;
  a.lse2 = w.lse2;
  a.Dvec = w.Dvec;
  a.dq_acc = w.acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = status;
  a.N = p.N;
  a.n_pad = w.n_pad;
  a.BH = p.B * p.H;
  a.causal = p.causal ? 1 : 0;
  a.window = p.window;
  a.n_blocks = w.n_pad / kBlk;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.drop = p.drop;
  return a;
}

template <int D, int DV, bool kDrop = false>
bool launch_seq(long long grid, int slot, const CUtensorMap& mq, const CUtensorMap& mk,
                const CUtensorMap& mv, const CUtensorMap& mdo, const BwdArgs& a, cudaStream_t stream) {
  using C = wide::BwdCfg<D, DV>;
  auto kern = wide::fa_bwd_main_seq<D, DV, kDrop>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes, slot)) return false;
  if (launch_overlapped(kern, dim3(static_cast<unsigned>(grid)), dim3(wide::kThreads), C::kSmemBytes, stream,
                        mq, mk, mv, mdo, a) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return true;
}

int launch_main_any(const Problem& p, const void* dO, void* dk, void* dv, void* workspace,
                    cudaStream_t stream) {
  const Workspace w = carve(p, workspace);
  const int BH = p.B * p.H;
  int* status = device_status_word();
  if (!status) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mdo;
  const int dvh = p.dv ? p.dv : p.d;
  if (!make_map_bhnd(&mq, p.q, BH, p.N, p.d) || !make_map_bhnd(&mk, p.k, BH, p.N, p.d) ||
      !make_map_bhnd(&mv, p.v, BH, p.N, dvh) || !make_map_bhnd(&mdo, dO, BH, p.N, dvh))
    return FA_ERR_LAUNCH;
  const BwdArgs a = make_args(p, w, dk, dv, status);
  const long long grid = static_cast<long long>(a.n_blocks) * BH;
  if (grid > 0x7fffffffLL) return FA_ERR_INVALID;
  if (p.drop.t > 0 && !(p.d == dvh && p.window == 0)) return FA_ERR_UNSUPPORTED;
  if (p.d == 64 && dvh == 64) {
    // persistent: one CTA per SM walks its share of the (key block, batch-head) items
    auto kern = p.drop.t > 0 ? pipe::fa_bwd_main_d64<true> : pipe::fa_bwd_main_d64<false>;
    if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), pipe::kSmemBytes, p.drop.t > 0 ? 12 : 2))
      return FA_ERR_LAUNCH;
    const int sms = device_sm_count();
    if (sms <= 0) return FA_ERR_LAUNCH;
    const long long g = grid < sms ? grid : sms;
    if (launch_overlapped(kern, dim3(static_cast<unsigned>(g)), dim3(pipe::kThreads), pipe::kSmemBytes,
                          stream, mq, mk, mv, mdo, a) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
  } else if (p.d == 128 && dvh == 128) {
    const bool ok = p.drop.t > 0 ? launch_seq<128, 128, true>(grid, 13, mq, mk, mv, mdo, a, stream)
                                 : launch_seq<128, 128>(grid, 3, mq, mk, mv, mdo, a, stream);
    if (!ok) return FA_ERR_LAUNCH;
  } else if (p.d == 128 && dvh == 64) {
    if (!launch_seq<128, 64>(grid, 6, mq, mk, mv, mdo, a, stream)) return FA_ERR_LAUNCH;
  } else if (p.d == 64 && dvh == 128) {
    if (!launch_seq<64, 128>(grid, 7, mq, mk, mv, mdo, a, stream)) return FA_ERR_LAUNCH;
  } else {
    return FA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

size_t bwd_workspace_bytes(long long B, long long H, long long N, long long d) {
  const long long n_pad = (N + kBlk - 1) / kBlk * kBlk;
  return static_cast<size_t>(2 * B * H * n_pad) * 4 + static_cast<size_t>(B * H * n_pad * d) * 4;
}

int launch_bwd_pre(const Problem& p, const void* o, const float* lse, const void* dO,
                   void* workspace, cudaStream_t stream) {
  const int dv = p.dv ? p.dv : p.d;
  if (p.d == 64 && dv == 64) return launch_pre_d<64, 64>(p, o, lse, dO, workspace, stream);
  if (p.d == 128 && dv == 128) return launch_pre_d<128, 128>(p, o, lse, dO, workspace, stream);
  if (p.d == 128 && dv == 64) return launch_pre_d<64, 128>(p, o, lse, dO, workspace, stream);
  if (p.d == 64 && dv == 128) return launch_pre_d<128, 64>(p, o, lse, dO, workspace, stream);
  return FA_ERR_UNSUPPORTED;
}

int launch_bwd_main(const Problem& p, const void* dO, void* dk, void* dv, void* workspace,
                    cudaStream_t stream) {
  const int dvh = p.dv ? p.dv : p.d;
  if ((p.d != 64 && p.d != 128) || (dvh != 64 && dvh != 128)) return FA_ERR_UNSUPPORTED;
  return launch_main_any(p, dO, dk, dv, workspace, stream);
}

int launch_bwd_post(const Problem& p, void* dq, const void* workspace, cudaStream_t stream) {
  const Workspace w = carve(p, const_cast<void*>(workspace));
  const int BH = p.B * p.H;
  const unsigned gy = BH < 65535 ? BH : 65535;
  cudaError_t e = cudaSuccess;
  if (p.d == 64) {
    const dim3 grid((p.N + 31) / 32, gy);
    e = launch_overlapped(fa_bwd_post<64>, grid, dim3(256), 0, stream, static_cast<const float*>(w.acc),
                          static_cast<uint4*>(dq), p.N, w.n_pad, BH);
  } else if (p.d == 128) {
    const dim3 grid((p.N + 15) / 16, gy);
    e = launch_overlapped(fa_bwd_post<128>, grid, dim3(256), 0, stream, static_cast<const float*>(w.acc),
                          static_cast<uint4*>(dq), p.N, w.n_pad, BH);
  } else {
    return FA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess && e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace fa
