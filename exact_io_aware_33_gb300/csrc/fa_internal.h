// Host-side declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

// Dropout on the attention probabilities (inactive when t = 0): an element
// is kept when its generator byte is >= t; kept values are scaled by
// inv_keep = 256 / (256 - t).
struct Dropout {
  uint32_t t = 0;
  float inv_keep = 1.0f;
  uint32_t seed_lo = 0, seed_hi = 0;
  uint32_t offset = 0;
};

// Problem description after argument checks.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  int B, H, N, d;
  int causal;
  float scale;
  int window = 0;  // backward only: 0 = none, else a causal window of this many keys
  int dv = 0;      // head size of V, O, dO and dV; 0 means d
  Dropout drop{};
};

// Forward problem with Nq queries over Nk keys (causal queries are the last
// Nq positions), head sizes d (Q, K) and dv (V, O), and an optional left
// window of `window` keys.
struct FwdProblem {
  const void* q;
  const void* k;
  const void* v;
  int B, H, Nq, Nk, d, dv;
  int causal;
  int window;
  float scale;
  Dropout drop{};
};

// Encodes a 3-D tiled TMA map over a bf16 [BH, N, d] tensor with boxes of
// box_rows rows x 64 columns and 128-byte swizzle. Returns false on failure.
bool make_map_bhnd(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows = 128);

// Size and scale checks shared by the entry points taking (B, H, N, d):
// FA_OK or an error code; *empty is set when there is nothing to compute.
int check_problem(int B, int H, int N, int d, float scale, bool* empty);

// FA_OK when the current device is a CC 10.3 GPU, else the error code.
int current_device_status();

// Device pointer of the status word of the current device (nullptr on error).
int* device_status_word();

// Number of SMs of the current device (looked up once per device), or 0.
int device_sm_count();

// Sets the dynamic shared memory limit of `func` once per device.
bool ensure_smem_attr(const void* func, int bytes, int slot);

// Launches `kern` on `stream` with programmatic stream serialization allowed:
// its CTAs may be scheduled, and run their set-up, while the previous kernel
// on the stream finishes; each kernel waits for that kernel
// (griddepcontrol.wait) before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem_bytes,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

int launch_fwd(const Problem& p, void* o, float* lse, cudaStream_t stream);
// part_o / part_lse == nullptr: one pass over the whole key range writing o and
// lse; otherwise the key range is split into n_splits parts whose fp32 states
// go to part_o [splits, BH, Nq, d] and part_lse [splits, BH, Nq] and are then
// merged into o and lse.
int launch_fwd_general(const FwdProblem& p, void* o, float* lse, float* part_o, float* part_lse,
                       int n_splits, cudaStream_t stream);
// The number of splits a split launch uses (n_splits <= 0: chosen from the
// problem size and the SM count).
int fwd_split_count(const FwdProblem& p, int n_splits, int sms);
int launch_bwd_pre(const Problem& p, const void* o, const float* lse, const void* dO,
                   void* workspace, cudaStream_t stream);
int launch_bwd_main(const Problem& p, const void* dO, void* dk, void* dv, void* workspace,
                    cudaStream_t stream);
int launch_bwd_post(const Problem& p, void* dq, const void* workspace, cudaStream_t stream);

size_t bwd_workspace_bytes(long long B, long long H, long long N, long long d);

}  // namespace fa
