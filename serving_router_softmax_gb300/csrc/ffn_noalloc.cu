// moe_verify_ffn_noalloc: the expert FFN with its scratch in a static device
// array, for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: code that runs while a
// CUDA graph is being captured (where cudaMalloc is not allowed), plugin or
// custom-op hosts that own the device allocator and forbid outside
// allocations, and latency-critical serving loops where an allocation would
// synchronise the device.  This entry point serves them by carving the FFN's
// scratch out of one file-scope array that is part of the loaded module.
//
// Trade-offs, stated for users:
//   * The array is kMaxScratchBytes (64 MiB) on every GPU that loads the
//     library, held until the process exits.
//   * All calls on a device share it and it keeps the previous call's
//     contents; the kernels clear what must start at zero on every call.
//     Calls that overlap on the GPU (different streams without ordering)
//     race on the array and give wrong results.
//   * The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture.  The address belongs to the device's
//     current context: after a context reset (cudaDeviceReset, or a host
//     framework recreating the primary context) the module is loaded again
//     and the array may move, so the next call on that device looks it up
//     again, and that call too should come before any capture.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kMaxScratchBytes = 64ull << 20;

static __device__ __align__(256) unsigned char g_ffn_scratch[kMaxScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};

// The current driver context (the identity of the loaded module's copy).
bool current_context(CUcontext* ctx) {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
  }
  return fn(ctx) == CUDA_SUCCESS && *ctx != nullptr;
}

// Device address of the scratch array on the current device, looked up once
// per device and context.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  void* p = nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  CUcontext ctx = nullptr;
  const bool have_ctx = current_context(&ctx);
  if (!g_scratch_ptr[dev] || !have_ctx || ctx != g_scratch_ctx[dev]) {
    if (cudaGetSymbolAddress(&p, g_ffn_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    // the context exists now (the lookup makes the runtime create it if needed)
    g_scratch_ctx[dev] = current_context(&ctx) ? ctx : nullptr;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_verify_ffn_noalloc(const void* x, int32_t T, int32_t k, const moe_layer_weights* lw,
                                      const int32_t* n_unique, const int32_t* unique,
                                      const int32_t* offsets, const int32_t* perm_token,
                                      const int32_t* inv, const float* w, float* y, int32_t* dev_err,
                                      void* stream) {
  using namespace moe;
  if (!lw) return MOE_ERR_ARG;
  int st = ffn_validate(*lw, T, k);
  if (st != MOE_OK) return st;
  if (T > 0 && (!x || !n_unique || !unique || !offsets || !perm_token || !inv || !w || !y))
    return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  const size_t need = ffn_workspace_bytes(*lw, T, k);
  if (need > kMaxScratchBytes) return MOE_ERR_UNSUPPORTED;  // beyond the static scratch
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != MOE_OK) return st;
  FfnArgs a{x, nullptr, 0, T, k, *lw, n_unique, unique, offsets, perm_token, inv, w, y,
            scratch, kMaxScratchBytes, dev_err, static_cast<cudaStream_t>(stream)};
  return ffn_launch(a);
}
