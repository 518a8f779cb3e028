// Host-side declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

// Problem description after argument checks.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  int B, H, N, d;
  int causal;
  float scale;
};

// Encodes a 3-D tiled TMA map over a bf16 [BH, N, d] tensor with boxes of
// 128 rows x 64 columns and 128-byte swizzle. Returns false on failure.
bool make_map_bhnd(CUtensorMap* map, const void* ptr, int BH, int N, int d);

// FA_OK when the current device is a CC 10.3 GPU, else the error code.
int current_device_status();

// Device pointer of the status word of the current device (nullptr on error).
int* device_status_word();

// Sets the dynamic shared memory limit of `func` once per device.
bool ensure_smem_attr(const void* func, int bytes, int slot);

int launch_fwd(const Problem& p, void* o, float* lse, cudaStream_t stream);
int launch_bwd_pre(const Problem& p, const void* o, const float* lse, const void* dO,
                   void* workspace, cudaStream_t stream);
int launch_bwd_main(const Problem& p, const void* dO, void* dk, void* dv, void* workspace,
                    cudaStream_t stream);
int launch_bwd_post(const Problem& p, void* dq, const void* workspace, cudaStream_t stream);

size_t bwd_workspace_bytes(long long B, long long H, long long N, long long d);

}  // namespace fa
