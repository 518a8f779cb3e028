// C ABI of libfa.so: argument checks, TMA tensor maps, the device status
// word, and the extern "C" entry points declared in fa.h.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// One status word per device: set by a kernel whose bounded wait ran out.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSmemSlots = 20;

struct DeviceState {
  bool probed = false;
  bool supported = false;
  int sms = 0;
  int* status = nullptr;
  bool smem_set[kSmemSlots] = {};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// Current device, checked once: compute capability 10.3 (GB300).
int current_device(DeviceState** st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_LAUNCH;
    s.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_LAUNCH;
    void* addr = nullptr;
    if (s.supported) {
      if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return FA_ERR_LAUNCH;
      s.status = static_cast<int*>(addr);
    }
    s.probed = true;
  }
  *st = &s;
  return s.supported ? FA_OK : FA_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Common checks of both passes. Returns FA_OK, or an error code; sets
// *empty when there is nothing to compute.
int check_problem(int B, int H, int N, int d, float scale, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) {
    *empty = true;
    return FA_OK;
  }
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 31) - 1) return FA_ERR_INVALID;
  // TMA coordinates and tensor extents are 32-bit; keep element offsets in range.
  if (bh * static_cast<long long>(N) * d > (1LL << 46)) return FA_ERR_INVALID;
  return FA_OK;
}

bool make_map_bhnd(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int current_device_status() {
  DeviceState* st = nullptr;
  return current_device(&st);
}

int* device_status_word() {
  DeviceState* st = nullptr;
  if (current_device(&st) != FA_OK) return nullptr;
  return st->status;
}

int device_sm_count() {
  DeviceState* st = nullptr;
  if (current_device(&st) != FA_OK) return 0;
  return st->sms;
}

bool ensure_smem_attr(const void* func, int bytes, int slot) {
  DeviceState* st = nullptr;
  if (current_device(&st) != FA_OK || slot < 0 || slot >= kSmemSlots) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!st->smem_set[slot]) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
      return false;
    st->smem_set[slot] = true;
  }
  return true;
}

}  // namespace fa

using fa::Problem;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_INVALID: return "invalid argument (pointer, size, alignment or scale)";
    case FA_ERR_UNSUPPORTED:
      return "unsupported (head size 64 or 128, or 256 in the forward; device must be CC 10.3)";
    case FA_ERR_LAUNCH: return "a CUDA call failed (launch, attribute or tensor map)";
    case FA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown error code";
  }
}

int fa_fwd_stream(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int N, int d, int causal, float scale, void* cuda_stream) {
  bool empty = false;
  int rc = fa::check_problem(B, H, N, d, scale, &empty);
  if (rc != FA_OK || empty) return rc;
  if (!fa::aligned16(q) || !fa::aligned16(k) || !fa::aligned16(v) || !fa::aligned16(o) ||
      !fa::aligned16(lse))
    return FA_ERR_INVALID;
  fa::DeviceState* st = nullptr;
  rc = fa::current_device(&st);
  if (rc != FA_OK) return rc;
  Problem p{q, k, v, B, H, N, d, causal, scale};
  return fa::launch_fwd(p, o, lse, static_cast<cudaStream_t>(cuda_stream));
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale) {
  return fa_fwd_stream(q, k, v, o, lse, B, H, N, d, causal, scale, nullptr);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  return fa::bwd_workspace_bytes(B, H, N, d);
}

namespace {

// Checks shared by the backward entry points. `ptrs` must all be non-NULL
// and 16-byte aligned; the workspace 256-byte aligned and large enough.
int check_bwd(int B, int H, int N, int d, float scale, std::initializer_list<const void*> ptrs,
              const void* workspace, size_t ws_bytes, bool* empty) {
  int rc = fa::check_problem(B, H, N, d, scale, empty);
  if (rc != FA_OK || *empty) return rc;
  if (d == 256) return FA_ERR_UNSUPPORTED;  // the backward's accumulators need d <= 128
  for (const void* ptr : ptrs)
    if (!fa::aligned16(ptr)) return FA_ERR_INVALID;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      ws_bytes < fa::bwd_workspace_bytes(B, H, N, d))
    return FA_ERR_WORKSPACE;
  fa::DeviceState* st = nullptr;
  return fa::current_device(&st);
}

}  // namespace

int fa_bwd_preprocess_stream(const void* o, const float* lse, const void* dO, int B, int H,
                             int N, int d, void* workspace, size_t ws_bytes, void* cuda_stream) {
  bool empty = false;
  int rc = check_bwd(B, H, N, d, 1.f, {o, lse, dO}, workspace, ws_bytes, &empty);
  if (rc != FA_OK || empty) return rc;
  Problem p{nullptr, nullptr, nullptr, B, H, N, d, 0, 1.f};
  return fa::launch_bwd_pre(p, o, lse, dO, workspace, static_cast<cudaStream_t>(cuda_stream));
}

int fa_bwd_main_stream(const void* q, const void* k, const void* v, const void* dO, void* dk,
                       void* dv, int B, int H, int N, int d, int causal, float scale,
                       void* workspace, size_t ws_bytes, void* cuda_stream) {
  bool empty = false;
  int rc = check_bwd(B, H, N, d, scale, {q, k, v, dO, dk, dv}, workspace, ws_bytes, &empty);
  if (rc != FA_OK || empty) return rc;
  Problem p{q, k, v, B, H, N, d, causal, scale};
  return fa::launch_bwd_main(p, dO, dk, dv, workspace, static_cast<cudaStream_t>(cuda_stream));
}

int fa_bwd_finish_stream(void* dq, int B, int H, int N, int d, const void* workspace,
                         size_t ws_bytes, void* cuda_stream) {
  bool empty = false;
  int rc = check_bwd(B, H, N, d, 1.f, {dq}, workspace, ws_bytes, &empty);
  if (rc != FA_OK || empty) return rc;
  Problem p{nullptr, nullptr, nullptr, B, H, N, d, 0, 1.f};
  return fa::launch_bwd_post(p, dq, workspace, static_cast<cudaStream_t>(cuda_stream));
}

int fa_bwd_stream(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, float scale, void* workspace, size_t ws_bytes, void* cuda_stream) {
  bool empty = false;
  int rc = check_bwd(B, H, N, d, scale, {q, k, v, o, lse, dO, dq, dk, dv}, workspace, ws_bytes,
                     &empty);
  if (rc != FA_OK || empty) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  Problem p{q, k, v, B, H, N, d, causal, scale};
  rc = fa::launch_bwd_pre(p, o, lse, dO, workspace, st);
  if (rc == FA_OK) rc = fa::launch_bwd_main(p, dO, dk, dv, workspace, st);
  if (rc == FA_OK) rc = fa::launch_bwd_post(p, dq, workspace, st);
  return rc;
}

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
              int d_v, int causal, int window, float scale, void* workspace, size_t ws_bytes,
              void* cuda_stream) {
  if (window < 0 || (window > 0 && !causal)) return FA_ERR_INVALID;
  if (d_v != 64 && d_v != 128) return FA_ERR_UNSUPPORTED;
  bool empty = false;
  int rc = check_bwd(B, H, N, d, scale, {q, k, v, o, lse, dO, dq, dk, dv}, workspace, ws_bytes,
                     &empty);
  if (rc != FA_OK || empty) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  Problem p{q, k, v, B, H, N, d, causal, scale, window, d_v};
  rc = fa::launch_bwd_pre(p, o, lse, dO, workspace, st);
  if (rc == FA_OK) rc = fa::launch_bwd_main(p, dO, dk, dv, workspace, st);
  if (rc == FA_OK) rc = fa::launch_bwd_post(p, dq, workspace, st);
  return rc;
}

namespace {

// Dropout parameters after checks: FA_ERR_INVALID unless 0 <= p < 1.
int make_dropout(float p, unsigned long long seed, unsigned long long offset, fa::Dropout* out) {
  if (!(p >= 0.f && p < 1.f)) return FA_ERR_INVALID;
  long t = lrintf(256.f * p);
  if (t > 255) t = 255;
  out->t = static_cast<uint32_t>(t);
  out->inv_keep = 256.f / static_cast<float>(256 - t);
  out->seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
  out->seed_hi = static_cast<uint32_t>(seed >> 32);
  out->offset = static_cast<uint32_t>(offset & 0xffffffffull);
  return FA_OK;
}

}  // namespace

int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, int causal, float scale, float dropout_p, unsigned long long seed,
                   unsigned long long offset, void* cuda_stream) {
  fa::Dropout drop;
  int rc = make_dropout(dropout_p, seed, offset, &drop);
  if (rc != FA_OK) return rc;
  bool empty = false;
  rc = fa::check_problem(B, H, N, d, scale, &empty);
  if (rc != FA_OK || empty) return rc;
  if (!fa::aligned16(q) || !fa::aligned16(k) || !fa::aligned16(v) || !fa::aligned16(o) ||
      !fa::aligned16(lse))
    return FA_ERR_INVALID;
  fa::DeviceState* st = nullptr;
  rc = fa::current_device(&st);
  if (rc != FA_OK) return rc;
  Problem p{q, k, v, B, H, N, d, causal, scale};
  p.drop = drop;
  return fa::launch_fwd(p, o, lse, static_cast<cudaStream_t>(cuda_stream));
}

int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, float dropout_p, unsigned long long seed,
                   unsigned long long offset, void* workspace, size_t ws_bytes, void* cuda_stream) {
  fa::Dropout drop;
  int rc = make_dropout(dropout_p, seed, offset, &drop);
  if (rc != FA_OK) return rc;
  bool empty = false;
  rc = check_bwd(B, H, N, d, scale, {q, k, v, o, lse, dO, dq, dk, dv}, workspace, ws_bytes, &empty);
  if (rc != FA_OK || empty) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  Problem p{q, k, v, B, H, N, d, causal, scale};
  p.drop = drop;
  rc = fa::launch_bwd_pre(p, o, lse, dO, workspace, st);
  if (rc == FA_OK) rc = fa::launch_bwd_main(p, dO, dk, dv, workspace, st);
  if (rc == FA_OK) rc = fa::launch_bwd_post(p, dq, workspace, st);
  return rc;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
           float scale) {
  bool empty = false;
  int rc = fa::check_problem(B, H, N, d, scale, &empty);
  if (rc != FA_OK || empty) return rc;
  if (d == 256) return FA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!fa::aligned16(ptr)) return FA_ERR_INVALID;
  fa::DeviceState* st = nullptr;
  rc = fa::current_device(&st);
  if (rc != FA_OK) return rc;
  const size_t bytes = fa::bwd_workspace_bytes(B, H, N, d);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, nullptr) != cudaSuccess) return FA_ERR_LAUNCH;
  rc = fa_bwd_stream(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, ws, bytes,
                     nullptr);
  if (cudaFreeAsync(ws, nullptr) != cudaSuccess && rc == FA_OK) rc = FA_ERR_LAUNCH;
  return rc;
}

namespace {

// Checks of the extended forward forms; sets *empty for B, H or Nq = 0.
int check_fwd_ex(int B, int H, int Nq, int Nk, int d, int dv, int causal, int window, float scale,
                 std::initializer_list<const void*> ptrs, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || window < 0) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID;
  // (d, dv) in {64, 128}^2, or d = dv = 256
  if (!(d == 256 && dv == 256) && ((d != 64 && d != 128) || (dv != 64 && dv != 128)))
    return FA_ERR_UNSUPPORTED;
  if (window > 0 && !causal) return FA_ERR_INVALID;
  if (B == 0 || H == 0 || Nq == 0) {
    *empty = true;
    return FA_OK;
  }
  if (Nk == 0 || (causal && Nq > Nk)) return FA_ERR_INVALID;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 31) - 1) return FA_ERR_INVALID;
  if (bh * static_cast<long long>(Nq > Nk ? Nq : Nk) * (d > dv ? d : dv) > (1LL << 46))
    return FA_ERR_INVALID;
  for (const void* ptr : ptrs)
    if (!fa::aligned16(ptr)) return FA_ERR_INVALID;
  fa::DeviceState* st = nullptr;
  return fa::current_device(&st);
}

int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

}  // namespace

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, int dv, int causal, int window, float scale,
              void* cuda_stream) {
  bool empty = false;
  int rc = check_fwd_ex(B, H, Nq, Nk, d, dv, causal, window, scale, {q, k, v, o, lse}, &empty);
  if (rc != FA_OK || empty) return rc;
  fa::FwdProblem p{q, k, v, B, H, Nq, Nk, d, dv, causal, window, scale};
  return fa::launch_fwd_general(p, o, lse, nullptr, nullptr, 1,
                                static_cast<cudaStream_t>(cuda_stream));
}

int fa_decode_num_splits(int B, int H, int Nq, int Nk, int n_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return 0;
  fa::FwdProblem p{nullptr, nullptr, nullptr, B, H, Nq, Nk, 64, 64, 0, 0, 1.f};
  return fa::fwd_split_count(p, n_splits, sm_count());
}

size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int dv, int n_splits) {
  const int s = fa_decode_num_splits(B, H, Nq, Nk, n_splits);
  if (s <= 0 || dv <= 0) return 0;
  return static_cast<size_t>(s) * B * H * Nq * (static_cast<size_t>(dv) + 1) * 4;
}

int fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, int dv, int causal, int window, float scale,
                      int n_splits, void* workspace, size_t ws_bytes, void* cuda_stream) {
  bool empty = false;
  int rc = check_fwd_ex(B, H, Nq, Nk, d, dv, causal, window, scale, {q, k, v, o, lse}, &empty);
  if (rc != FA_OK || empty) return rc;
  const size_t need = fa_decode_workspace_bytes(B, H, Nq, Nk, dv, n_splits);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < need)
    return FA_ERR_WORKSPACE;
  const int s = fa_decode_num_splits(B, H, Nq, Nk, n_splits);
  fa::FwdProblem p{q, k, v, B, H, Nq, Nk, d, dv, causal, window, scale};
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = part_o + static_cast<size_t>(s) * B * H * Nq * dv;
  return fa::launch_fwd_general(p, o, lse, part_o, part_lse, s,
                                static_cast<cudaStream_t>(cuda_stream));
}

int fa_get_last_device_status(void) {
  fa::DeviceState* st = nullptr;
  if (fa::current_device(&st) != FA_OK) return FA_ERR_LAUNCH;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_LAUNCH;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_status_word, sizeof(int)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const int zero = 0;
  if (cudaMemcpyToSymbol(fa::g_status_word, &zero, sizeof(int)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return word == fa::kStatusTimeout ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
