// Backward pass of exact attention on sm_103a (placeholder until the
// recompute kernels land).
#include "fa.h"
#include "fa_internal.h"

namespace fa {

size_t bwd_workspace_bytes(long long B, long long H, long long N, long long d) {
  // D (fp32 [B,H,N]) followed by the fp32 dQ accumulator ([B,H,N,d]).
  const size_t d_bytes = static_cast<size_t>(B * H * N) * 4;
  const size_t d_pad = (d_bytes + 255) & ~static_cast<size_t>(255);
  return d_pad + static_cast<size_t>(B * H * N * d) * 4;
}

int launch_bwd(const Problem&, const void*, const float*, const void*, void*, void*, void*, void*,
               cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
