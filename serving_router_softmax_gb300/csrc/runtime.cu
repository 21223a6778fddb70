// Library runtime: status strings, launch accounting and optional per-kernel
// event timing.
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {
namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_test_stall{0};
std::atomic<int> g_nvtx{0};

struct Prof {
  std::mutex mu;
  bool on = false;
  int max = 0;
  std::vector<cudaEvent_t> ev;   // 2 per record
  std::vector<int> cls;
  int n = 0;
  int pending_cls = -1;
  int mask = 0;
};
Prof& prof() {
  static Prof p;
  return p;
}

}  // namespace

int test_stall_mask() { return g_test_stall.load(std::memory_order_relaxed); }

NvtxRange::NvtxRange(const char* name) : on(g_nvtx.load(std::memory_order_relaxed) != 0) {
  if (on) nvtxRangePushA(name);
}
NvtxRange::~NvtxRange() {
  if (on) nvtxRangePop();
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

void note_launch(int c, cudaStream_t s, bool before) {
  if (!before) g_launches.fetch_add(1, std::memory_order_relaxed);
  Prof& p = prof();
  if (!p.on) return;
  std::lock_guard<std::mutex> lk(p.mu);
  if (!p.on) return;
  if (!((p.mask >> c) & 1)) return;
  if (before) {
    if (p.n >= p.max) return;
    cudaEventRecord(p.ev[2 * p.n], s);
    p.pending_cls = c;
  } else {
    if (p.n >= p.max || p.pending_cls != c) return;
    cudaEventRecord(p.ev[2 * p.n + 1], s);
    p.cls[p.n] = c;
    ++p.n;
    p.pending_cls = -1;
  }
}

}  // namespace moe

extern "C" int moe_profile_begin(int32_t max_launches, int32_t class_mask) {
  using namespace moe;
  if (max_launches < 1 || max_launches > (1 << 20)) return MOE_ERR_ARG;
  Prof& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  for (auto e : p.ev) cudaEventDestroy(e);
  p.ev.assign(2 * static_cast<size_t>(max_launches), nullptr);
  for (auto& e : p.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
  p.cls.assign(max_launches, -1);
  p.max = max_launches;
  p.n = 0;
  p.pending_cls = -1;
  p.mask = class_mask;
  p.on = true;
  return MOE_OK;
}

extern "C" int moe_profile_end(float* ms_per_class, int32_t* launches_per_class, int32_t n_classes) {
  using namespace moe;
  Prof& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  if (!p.on) return MOE_ERR_ARG;
  p.on = false;
  for (int c = 0; c < n_classes; ++c) {
    if (ms_per_class) ms_per_class[c] = 0.f;
    if (launches_per_class) launches_per_class[c] = 0;
  }
  int st = MOE_OK;
  for (int i = 0; i < p.n; ++i) {
    if (cudaEventSynchronize(p.ev[2 * i + 1]) != cudaSuccess) {
      st = MOE_ERR_CUDA;
      break;
    }
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.ev[2 * i], p.ev[2 * i + 1]) != cudaSuccess) {
      st = MOE_ERR_CUDA;
      break;
    }
    int c = p.cls[i];
    if (c >= 0 && c < n_classes) {
      if (ms_per_class) ms_per_class[c] += ms;
      if (launches_per_class) launches_per_class[c] += 1;
    }
  }
  for (auto e : p.ev) cudaEventDestroy(e);
  p.ev.clear();
  p.n = 0;
  return st;
}

extern "C" const char* moe_status_str(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case MOE_ERR_CUDA: return "CUDA launch error";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

extern "C" uint64_t moe_launch_count(void) { return moe::g_launches.load(); }

extern "C" int moe_test_set_stall(int32_t mask) {
  if (mask & ~(MOE_TEST_STALL_GATE_UP | MOE_TEST_STALL_READY_FLAG)) return MOE_ERR_ARG;
  moe::g_test_stall.store(mask, std::memory_order_relaxed);
  return MOE_OK;
}

extern "C" int moe_set_nvtx(int32_t on) {
  if (on != 0 && on != 1) return MOE_ERR_ARG;
  moe::g_nvtx.store(on, std::memory_order_relaxed);
  return MOE_OK;
}

extern "C" int moe_version(void) { return 103; }
