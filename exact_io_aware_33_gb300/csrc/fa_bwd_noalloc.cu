// fa_bwd_noalloc: the backward pass with its scratch memory built into the
// library, for callers that cannot allocate device memory.
//
// fa_bwd needs a float32 workspace (D, the log2-domain LSE and the dQ
// accumulator). Most callers pass one (fa_bwd_stream) or let fa_bwd take it
// from cudaMallocAsync. Some callers can do neither: a host framework that
// owns every device allocation through its own allocator and forbids
// libraries to allocate behind its back, or a serving loop with a fixed
// memory budget that must never call cudaMalloc on its hot path (the call
// can synchronise the device and can fail once memory is fragmented). This
// entry point serves them: the workspace lives in a file-scope device array
// of fixed size, so the call allocates nothing.
//
// Costs and limits of that choice:
//   * the array is kScratchBytes (64 MiB). With lazy module loading (the
//     CUDA default) it is reserved on a device by the first call there: the
//     cudaGetSymbolAddress below loads this file's device code onto that
//     device. It stays reserved until the process exits. That first call can
//     fail when the device is full and must not run inside a stream capture,
//     so callers make it during set-up;
//   * problems whose workspace (fa_bwd_workspace_bytes) exceeds it are
//     rejected with FA_ERR_WORKSPACE before anything is launched;
//   * all calls share the one array: two calls whose kernels overlap on the
//     GPU (different streams, or several host threads) race and corrupt each
//     other's results. Serialise them on one stream.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kScratchBytes = FA_BWD_NOALLOC_MAX_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself. In host code this name is only a stand-in for the
// device symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached. nullptr on failure.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale,
                              void* cuda_stream) {
  // The size checks are fa_bwd_stream's own (check_problem), with the
  // built-in array standing in for the caller's workspace.
  bool empty = false;
  const int chk = fa::check_problem(B, H, N, d, scale, &empty);
  if (chk != FA_OK || empty) return chk;
  if (d == 256) return FA_ERR_UNSUPPORTED;  // as fa_bwd_stream: the backward takes d <= 128
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!fa::aligned16(ptr)) return FA_ERR_INVALID;
  if (fa::bwd_workspace_bytes(B, H, N, d) > fa::kScratchBytes) return FA_ERR_WORKSPACE;
  const int dev_rc = fa::current_device_status();
  if (dev_rc != FA_OK) return dev_rc;
  // First call on a device: finds the array's device address (and, with lazy
  // module loading, loads this file's device code there).
  void* ws = fa::scratch_on_current_device();
  if (ws == nullptr) return FA_ERR_LAUNCH;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  fa::Problem p{q, k, v, B, H, N, d, causal, scale};
  // The preprocess stage zeroes the dQ accumulator, so whatever the last
  // call left in the array does not leak into this one.
  int rc = fa::launch_bwd_pre(p, o, lse, dO, ws, st);
  if (rc == FA_OK) rc = fa::launch_bwd_main(p, dO, dk, dv, ws, st);
  if (rc == FA_OK) rc = fa::launch_bwd_post(p, dq, ws, st);
  return rc;
}
