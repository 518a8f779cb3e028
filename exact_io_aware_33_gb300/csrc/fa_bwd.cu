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
//   fa_bwd_main  one CTA per (key/value block of 128 keys, batch-head): K_j
//                and V_j stay in shared memory and dK_j, dV_j accumulate in
//                tensor memory while the query blocks i stream past; per i
//                five tcgen05 MMAs:
//                  S^T  = K_j Q_i^T         (TMEM)
//                  dP^T = V_j dO_i^T        (TMEM)
//                  -> P^T, dS^T in registers (thread = key row)
//                  dV  += P^T dO_i          (P^T read from TMEM)
//                  dK  += dS^T Q_i          (dS^T read from shared memory)
//                  dQ_i = dS K_j            (same shared bytes, MN-major)
//                dQ_i is added into the fp32 accumulator in global memory.
//   fa_bwd_post  dQ = bf16(accumulator)
//
// CTA of fa_bwd_main (512 threads):
//   warps 0-7  two P/dS warpgroups: thread = key row = TMEM lane; warpgroup
//              w handles query columns [64w, 64w+64) of each step, and the
//              S^T / dP^T MMAs run one query half at a time, so the first
//              half's P/dS work overlaps the second half's MMAs
//   warps 8-11 dQ warpgroup: reads dQ_i (thread = query row) and adds it
//              into global memory; writes dK, dV at the end (thread = key)
//   warp  12   tcgen05 MMA issue and TMEM allocation
//   warp  13   TMA producer; warps 14-15 idle
//
// TMEM columns: S^T/P^T [0,128), dP^T [128,256); for d = 64 dQ [256,320),
// dK [320,384), dV [384,448); for d = 128 dQ reuses the dP^T columns (the
// next dP^T waits until dQ has been read), dK [256,384), dV [384,512).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBlk = 128;  // keys per CTA block and queries per step
constexpr int kHalf = 64;  // query columns per P/dS warpgroup
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kLoadWarp = 13;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kBlk * 64 * 2;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kVecBytes = 2 * kBlk * 4;  // lse2[128], D[128] of one query block
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr bool kDqAliasDp = (D == 128);
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kDSOff = kVOff + kTileBytes;             // 2 x 16 KiB
  static constexpr int kStageOff = kDSOff + 2 * kChunkBytes;
  static constexpr int kStageBytes = 2 * kTileBytes + kVecBytes;  // Q, dO, vectors
  static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = kBarQFull + kStages;
  static constexpr int kBarSFull = kBarQEmpty + kStages;    // one per query half
  static constexpr int kBarDSFull = kBarSFull + 2;           // one per query half
  static constexpr int kBarDQFull = kBarDSFull + 2;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarDKDV = kBarDQEmpty + 1;
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
};

struct BwdArgs {
  const float* lse2;   // [BH, Npad] -LSE * log2(e), -inf past N
  const float* Dvec;   // [BH, Npad] -rowsum(dO * O), 0 past N
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int N;
  int n_pad;
  int BH;
  int causal;
  int n_blocks;
  float scale;
  float scale_log2;
};

// ---------------------------------------------------------------- B0
// For every row of the padded [BH, Npad] grid: -D = -sum_c dO[c] * O[c] and
// -LSE * log2(e) (rows past N get 0 and -inf, so that their recomputed
// probabilities are exactly 0). Stored negated so the main kernel's packed
// FMAs take them as addends. One group of D/8 lanes per row, each lane
// reading 8 bf16 (16 bytes) of both tensors. Also zeroes dq_acc.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const __nv_bfloat16* __restrict__ o,
                                                  const __nv_bfloat16* __restrict__ dO,
                                                  const float* __restrict__ lse,
                                                  float* __restrict__ Dvec,
                                                  float* __restrict__ lse2, int N, int n_pad,
                                                  long long pad_rows, float4* __restrict__ dq_acc,
                                                  long long acc_vec4) {
  constexpr int kTpr = D / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;  // multiple of 32
  const long long tid0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long lanes = ((pad_rows * kTpr + 31) / 32) * 32;
  for (long long t = tid0; t < lanes; t += stride) {
    const long long prow = t / kTpr;
    const int sub = static_cast<int>(t % kTpr);
    const long long bh = prow / n_pad;
    const int n = static_cast<int>(prow - bh * n_pad);
    const bool live = prow < pad_rows && n < N;
    float acc = 0.f;
    if (live) {
      const long long row = bh * N + n;
      const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + sub * 8);
      const uint4 b = *reinterpret_cast<const uint4*>(dO + row * D + sub * 8);
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
    if (prow < pad_rows && sub == 0) {
      Dvec[prow] = -acc;
      lse2[prow] = live ? -lse[bh * N + n] * kLog2e : -INFINITY;
    }
  }
  for (long long i = tid0; i < acc_vec4; i += stride) dq_acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------- B2
__global__ void __launch_bounds__(256) fa_bwd_post(const float4* __restrict__ acc,
                                                   uint2* __restrict__ dq, long long n_vec4) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec4;
       i += stride) {
    const float4 a = acc[i];
    dq[i] = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
  }
}

// ---------------------------------------------------------------- B1
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const BwdArgs args) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kMiscOff + 4);
  if (base - raw_u32 + C::kLayoutBytes > static_cast<uint32_t>(C::kSmemBytes)) {
    // The dynamic shared memory base is not aligned enough for this layout.
    if (threadIdx.x == 0) atomicExch(args.status, kStatusTimeout);
    return;
  }

  const int N = args.N;
  const int bh = blockIdx.x % args.BH;
  const int jb = static_cast<int>(blockIdx.x / args.BH);  // key block (heaviest first)
  const int i0 = args.causal ? jb : 0;
  const int n_steps = args.n_blocks - i0;
  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarQFull + s), 1);
      mbar_init(bar(C::kBarQEmpty + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kBarSFull + h), 1);
      mbar_init(bar(C::kBarDSFull + h), 128);
    }
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQEmpty), 128);
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

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmDO);
      mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(base + C::kKOff + c * C::kChunkBytes, &tmK, bar(C::kBarKV), c * 64, jb * kBlk, bh);
        tma_load_3d(base + C::kVOff + c * C::kChunkBytes, &tmV, bar(C::kBarKV), c * 64, jb * kBlk, bh);
      }
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n_steps; ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages)
          ok = mbar_wait(bar(C::kBarQEmpty + s), ((it / C::kStages) + 1) & 1, abort_flag);
        if (!ok) break;
        const int row0 = (i0 + it) * kBlk;
        const uint32_t st = base + C::kStageOff + s * C::kStageBytes;
        const uint32_t fb = bar(C::kBarQFull + s);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(st + c * C::kChunkBytes, &tmQ, fb, c * 64, row0, bh);
          tma_load_3d(st + C::kTileBytes + c * C::kChunkBytes, &tmDO, fb, c * 64, row0, bh);
        }
        const size_t voff = static_cast<size_t>(bh) * args.n_pad + row0;
        bulk_load(st + 2 * C::kTileBytes, args.lse2 + voff, kBlk * 4, fb);
        bulk_load(st + 2 * C::kTileBytes + kBlk * 4, args.Dvec + voff, kBlk * 4, fb);
        issued = it + 1;
      }
      if (*abort_flag) {
        mbar_wait(bar(C::kBarKV), 0, nullptr);
        for (int it = issued - 1; it >= 0 && it >= issued - C::kStages; --it)
          mbar_wait(bar(C::kBarQFull + it % C::kStages), (it / C::kStages) & 1, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdT = idesc_bf16_f32(kBlk, kHalf, false, false); // S^T, dP^T halves
      constexpr uint32_t kIdKV = idesc_bf16_f32(kBlk, D, false, true);     // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(kBlk, D, true, true);       // dQ
      const uint32_t kb = base + C::kKOff, vb = base + C::kVOff, dsb = base + C::kDSOff;
      bool ok = mbar_wait(bar(C::kBarKV), 0, abort_flag);
      tc_fence_after();
      for (int it = 0; it < n_steps && ok; ++it) {
        const int s = it % C::kStages;
        ok = mbar_wait(bar(C::kBarQFull + s), (it / C::kStages) & 1, abort_flag);
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
            mma_ss(tmem + C::kColS + kHalf * h, sdesc_sw128(kb + off, 16, 1024),
                   sdesc_sw128(qb + off + h * 8192, 16, 1024), kIdT, kk > 0 ? 1u : 0u);
          }
          if (C::kDqAliasDp && h == 0 && it > 0) {  // dQ of the last step shares dP's columns
            ok = mbar_wait(bar(C::kBarDQEmpty), (it - 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {  // dP^T_h = V dO_h^T
            const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            mma_ss(tmem + C::kColDP + kHalf * h, sdesc_sw128(vb + off, 16, 1024),
                   sdesc_sw128(dob + off + h * 8192, 16, 1024), kIdT, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBarSFull + h));
        }
        if (!ok) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          ok = mbar_wait(bar(C::kBarDSFull + h), it & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          // dV += P_h^T dO_h   (A = P^T in TMEM, B = dO rows of half h, MN-major)
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            mma_ts(tmem + C::kColDV, tmem + C::kColS + kHalf * h + kk * 8,
                   sdesc_sw128(dob + (4 * h + kk) * 2048, C::kChunkBytes, 1024), kIdKV,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
          // dK += dS_h^T Q_h   (A = dS^T K-major in smem region h, B = Q MN-major)
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            mma_ss(tmem + C::kColDK, sdesc_sw128(dsb + h * C::kChunkBytes + kk * 32, 16, 1024),
                   sdesc_sw128(qb + (4 * h + kk) * 2048, C::kChunkBytes, 1024), kIdKV,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        if (!C::kDqAliasDp && it > 0) {
          ok = mbar_wait(bar(C::kBarDQEmpty), (it - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
        }
        // dQ = dS K          (A = dS MN-major in smem, B = K MN-major)
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ss(tmem + C::kColDQ, sdesc_sw128(dsb + kk * 2048, C::kChunkBytes, 1024),
                 sdesc_sw128(kb + kk * 2048, C::kChunkBytes, 1024), kIdQ, kk > 0 ? 1u : 0u);
        mma_commit(bar(C::kBarDQFull));
        mma_commit(bar(C::kBarQEmpty + s));
      }
      if (ok) mma_commit(bar(C::kBarDKDV));
      mma_commit(bar(C::kBarDrain));
      mbar_wait(bar(C::kBarDrain), 0, nullptr);
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
    bool ok = true;
    for (int it = 0; it < n_steps; ++it) {
      const float* nlse2_s =
          reinterpret_cast<const float*>(base_ptr + C::kStageOff + (it % C::kStages) * C::kStageBytes +
                                         2 * C::kTileBytes) + kHalf * w;
      const float* nd_s = nlse2_s + kBlk;
      // the stage's vectors arrive with its Q/dO tiles; S^T, dP^T with the MMA commit
      ok = mbar_wait(bar(C::kBarQFull + it % C::kStages), (it / C::kStages) & 1, abort_flag);
      if (ok) ok = mbar_wait(bar(C::kBarSFull + w), it & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool diag = args.causal && it == 0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tS + c * 32, sr);
        tmem_ld32(tDP + c * 32, dr);
        tmem_ld_wait(sr);
        tmem_ld_wait(dr);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int ql = c * 32 + e;            // query column within this half
          const int qc = kHalf * w + ql;        // ... within the block
          const float2 nl = *reinterpret_cast<const float2*>(nlse2_s + ql);
          const float2 nd = *reinterpret_cast<const float2*>(nd_s + ql);
          const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                      sl2x2, nl);
          float2 p = make_float2(ex2(a.x), ex2(a.y));
          if (diag) {  // causal diagonal block: query before key is masked
            if (qc < key_row) p.x = 0.f;
            if (qc + 1 < key_row) p.y = 0.f;
          }
          const float2 g = __fmul2_rn(
              p, __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), nd));
          pp[e >> 1] = pack_bf16(p.x, p.y);
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
      mbar_arrive(bar(C::kBarDSFull + w));
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
      float* dst = args.dq_acc + (static_cast<size_t>(bh) * N + q) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t g[32];
        tmem_ld32(tmem + lane_base + C::kColDQ + c * 32, g);
        tmem_ld_wait(g);
        if (q < N) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            red_add_v4(dst + c * 32 + e, __uint_as_float(g[e]) * scale,
                       __uint_as_float(g[e + 1]) * scale, __uint_as_float(g[e + 2]) * scale,
                       __uint_as_float(g[e + 3]) * scale);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::kBarDQEmpty));
    }
    if (ok) {
      ok = mbar_wait(bar(C::kBarDKDV), 0, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const int key = jb * kBlk + r;
      const bool live = key < N;
      const size_t off = (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::kColDK : C::kColDV;
        const float mul = which == 0 ? scale : 1.f;
        __nv_bfloat16* out = (which == 0 ? args.dk : args.dv) + off;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t g[32];
          tmem_ld32(tmem + lane_base + col + c * 32, g);
          tmem_ld_wait(g);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(g[2 * e]) * mul, __uint_as_float(g[2 * e + 1]) * mul);
          if (live) {
            uint4* o4 = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) o4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(args.status, kStatusTimeout);
}

// Workspace sections: D and lse2 (fp32 [BH, Npad] each), then the fp32 dQ
// accumulator [BH, N, d]. Npad * 4 bytes is a multiple of 512, so every
// section and every query block's vector slice is 512-byte aligned.
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

template <int D>
int launch_pre_d(const Problem& p, const void* o, const float* lse, const void* dO,
                 void* workspace, cudaStream_t stream) {
  const Workspace w = carve(p, workspace);
  const long long acc_vec4 = static_cast<long long>(p.B) * p.H * p.N * D / 4;
  const long long work = w.pad_rows * (D / 8) > acc_vec4 ? w.pad_rows * (D / 8) : acc_vec4;
  long long blocks = (work + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  fa_bwd_pre<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, w.Dvec,
      w.lse2, p.N, w.n_pad, w.pad_rows, reinterpret_cast<float4*>(w.acc), acc_vec4);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

template <int D>
int launch_main_d(const Problem& p, const void* dO, void* dk, void* dv, void* workspace,
                  cudaStream_t stream) {
  using C = BwdCfg<D>;
  const Workspace w = carve(p, workspace);
  const int BH = p.B * p.H;
  int* status = device_status_word();
  if (!status) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_bhnd(&mq, p.q, BH, p.N, D) || !make_map_bhnd(&mk, p.k, BH, p.N, D) ||
      !make_map_bhnd(&mv, p.v, BH, p.N, D) || !make_map_bhnd(&mdo, dO, BH, p.N, D))
    return FA_ERR_LAUNCH;
  auto kern = fa_bwd_main<D>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes, D == 64 ? 2 : 3))
    return FA_ERR_LAUNCH;
  BwdArgs a;
  a.lse2 = w.lse2;
  a.Dvec = w.Dvec;
  a.dq_acc = w.acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = status;
  a.N = p.N;
  a.n_pad = w.n_pad;
  a.BH = BH;
  a.causal = p.causal ? 1 : 0;
  a.n_blocks = w.n_pad / kBlk;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  const long long grid = static_cast<long long>(a.n_blocks) * BH;
  if (grid > 0x7fffffffLL) return FA_ERR_INVALID;
  kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mdo, a);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

size_t bwd_workspace_bytes(long long B, long long H, long long N, long long d) {
  const long long n_pad = (N + kBlk - 1) / kBlk * kBlk;
  return static_cast<size_t>(2 * B * H * n_pad) * 4 + static_cast<size_t>(B * H * N * d) * 4;
}

int launch_bwd_pre(const Problem& p, const void* o, const float* lse, const void* dO,
                   void* workspace, cudaStream_t stream) {
  if (p.d == 64) return launch_pre_d<64>(p, o, lse, dO, workspace, stream);
  if (p.d == 128) return launch_pre_d<128>(p, o, lse, dO, workspace, stream);
  return FA_ERR_UNSUPPORTED;
}

int launch_bwd_main(const Problem& p, const void* dO, void* dk, void* dv, void* workspace,
                    cudaStream_t stream) {
  if (p.d == 64) return launch_main_d<64>(p, dO, dk, dv, workspace, stream);
  if (p.d == 128) return launch_main_d<128>(p, dO, dk, dv, workspace, stream);
  return FA_ERR_UNSUPPORTED;
}

int launch_bwd_post(const Problem& p, void* dq, const void* workspace, cudaStream_t stream) {
  const Workspace w = carve(p, const_cast<void*>(workspace));
  const long long acc_vec4 = static_cast<long long>(p.B) * p.H * p.N * p.d / 4;
  long long blocks = (acc_vec4 + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  fa_bwd_post<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(w.acc), static_cast<uint2*>(dq), acc_vec4);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace fa
