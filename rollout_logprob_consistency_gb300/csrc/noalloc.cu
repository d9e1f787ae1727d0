// tim_logprob_noalloc: the linear-logprob path with its scratch memory in a
// fixed device array owned by this library, for callers that cannot allocate
// device memory themselves.
//
// Who needs this: a scoring hook embedded in a rollout or serving engine that
// has already reserved nearly all free device memory for its own caches and
// pools (a cudaMalloc there fails, and the engine's allocator is not reachable
// from plain C), and latency-sensitive callers for whom cudaMalloc/cudaFree are
// off limits because they can synchronise the device.  Such callers pass their
// inputs and outputs only; the intermediate y, the per-vocabulary-tile records
// and the target logits live in the static array below.
//
// The array is a file-scope __device__ object: every GPU that loads the library
// holds kNoAllocScratchBytes of it until the process exits.  Host code must not
// hand the array's host-side name to a kernel (that name is a host stand-in,
// not a device address).  Set-up, once per CUDA context with that context
// current: fetch the device address with cudaGetSymbolAddress (this also places
// the library's module, and with it the array, on the device) and load every
// kernel the path can launch (the runtime loads kernels lazily, at first
// launch, and loading takes device memory).  The address is cached under the
// context's unique ID, so a context created after cudaDeviceReset gets its own
// set-up instead of a stale address.
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "tim_common.cuh"

namespace tim {
cudaError_t load_rmsnorm_rows_kernel();
cudaError_t load_scoring_gemm_kernels();
cudaError_t load_lse_finalize_kernel();
cudaError_t launch_rmsnorm_rows(const void* hidden, const void* gamma, int64_t T, int d, float eps,
                                void* y, int* status, cudaStream_t stream);
cudaError_t launch_lmhead_lse(const void* y, const void* W, const int32_t* ids, int64_t T, int d,
                              int V, float temperature, void* part, float* tgt, int* status,
                              cudaStream_t stream, int num_sms);
cudaError_t launch_lse_finalize(const void* part, const float* tgt, const int32_t* ids, int64_t T,
                                int V, float* out_lp, float* out_lse, int32_t* out_top1,
                                int* status, cudaStream_t stream);

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique ID of the current CUDA context (0 when none is current yet).  Drivers
// without cuCtxGetId get the context handle as the key instead (a new context may
// reuse a freed handle's value there, so the ID is preferred).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {  // called under g_addr_mutex
    void* p = nullptr;
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r1, r2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) !=
            cudaSuccess ||
        r1 != cudaDriverEntryPointSuccess)
      return false;
    get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) ==
            cudaSuccess &&
        r2 == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(q);
    cudaGetLastError();
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  if (ctx == nullptr) return true;
  if (get_id == nullptr) {
    *id = static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(ctx));
    return true;
  }
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context, with the set-up
// described above done the first time this context is seen on `dev`.
tim_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return TIM_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    cudaGetLastError();
    return TIM_ERR_CUDA;
  }
  if (id == 0 || g_addr[dev] == nullptr || g_ctx_id[dev] != id) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess) e = load_rmsnorm_rows_kernel();
    if (e == cudaSuccess) e = load_scoring_gemm_kernels();
    if (e == cudaSuccess) e = load_lse_finalize_kernel();
    if (e != cudaSuccess || p == nullptr || !current_context_id(&id) || id == 0) {
      cudaGetLastError();
      g_addr[dev] = nullptr;
      return TIM_ERR_CUDA;
    }
    g_addr[dev] = p;
    g_ctx_id[dev] = id;
  }
  *out = g_addr[dev];
  return TIM_OK;
}

inline bool is_aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace
}  // namespace tim

using namespace tim;

extern "C" tim_status tim_logprob_noalloc(const void* hidden, const void* gamma, const void* W,
                                          const int32_t* token_ids, int64_t T, int32_t d,
                                          int32_t V, float temperature, float eps,
                                          float* out_logprob, float* out_lse, int32_t* out_top1,
                                          int32_t* out_status, tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || W == nullptr || token_ids == nullptr ||
      out_logprob == nullptr || out_lse == nullptr || out_top1 == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!is_aligned(hidden, 16) || !is_aligned(gamma, 16) || !is_aligned(W, 16) ||
      !is_aligned(token_ids, 4) || !is_aligned(out_logprob, 4) || !is_aligned(out_lse, 4) ||
      !is_aligned(out_top1, 4) || (out_status != nullptr && !is_aligned(out_status, 4)))
    return TIM_ERR_INVALID_ARG;
  if (T < 1 || T > INT32_MAX || d < 64 || d > 65536 || (d % 64) != 0 || V < 1 ||
      V > INT32_MAX - 256)
    return TIM_ERR_SHAPE;
  if (!(std::isfinite(temperature) && temperature > 0.f) || !(std::isfinite(eps) && eps >= 0.f))
    return TIM_ERR_INVALID_ARG;
  const WsLayout L = logprob_layout(T, d, V);
  if (L.total > kNoAllocScratchBytes) return TIM_ERR_WORKSPACE;  // beyond the fixed scratch

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return TIM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return TIM_ERR_UNSUPPORTED_DEVICE;
  void* scratch = nullptr;
  tim_status s = scratch_address(dev, &scratch);
  if (s != TIM_OK) return s;

  uint8_t* base = static_cast<uint8_t*>(scratch);
  int* status = reinterpret_cast<int*>(base + L.status_off);
  void* y = base + L.y_off;
  void* part = base + L.part_off;
  float* tgt = reinterpret_cast<float*>(base + L.tgt_off);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  // The array keeps the previous call's bytes: only the status word must start
  // at zero (y, the records and the used target logits are written before read).
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return TIM_ERR_CUDA;
  if (launch_rmsnorm_rows(hidden, gamma, T, d, eps, y, status, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_lmhead_lse(y, W, token_ids, T, d, V, temperature, part, tgt, status, st, sms) !=
      cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_lse_finalize(part, tgt, token_ids, T, V, out_logprob, out_lse, out_top1, status,
                          st) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (out_status != nullptr &&
      cudaMemcpyAsync(out_status, status, sizeof(int), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return TIM_ERR_CUDA;
  return TIM_OK;
}
