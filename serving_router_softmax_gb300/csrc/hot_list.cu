// moe_hot_list: the hot-expert list of expert-level residency.
//
// S2-MoE write-up, "system implementation: expert-level offloading": with
// spare device memory, a list of frequently activated experts, found by
// offline profiling of activation frequencies, stays resident.  The reading
// applied here: count each expert's activations over the profiled routing
// decisions and keep the n_hot experts with the largest counts, equal counts
// going to the lower expert id.  The list is written in ascending id order,
// and hot expert j gets home slot first_slot + j (the pool layout of
// moe_expert_pool); every other expert's home slot is -1.
//
// One CTA: shared-memory integer counts (exact whatever the order of the
// atomics), a rank per expert against every other expert (the order is a
// strict total order, so ranks are distinct), and a block-wide prefix sum
// of the hot flags in id order.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kHotThreads = 1024;
constexpr int kHotMaxE = 4096;
constexpr int kPerThread = kHotMaxE / kHotThreads;  // consecutive experts per thread in the scan

struct HotArgs {
  const int32_t* ids;
  long long n_ids;
  int E, n_hot, first_slot;
  int32_t* counts;
  int32_t* hot;
  int32_t* home_slot;
  int32_t* dev_err;
};

__global__ void __launch_bounds__(kHotThreads) hot_list_kernel(const HotArgs a) {
  __shared__ int32_t cnt[kHotMaxE];
  __shared__ int32_t warp_tot[kHotThreads / kWarp];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int e = tid; e < a.E; e += kHotThreads) cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (long long i = tid; i < a.n_ids; i += kHotThreads) {
    const int e = a.ids[i];
    if (e == -1) continue;
    if (e < 0 || e >= a.E) {
      bad = true;
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  if (bad) flag_error(a.dev_err, MOE_DEV_BAD_ID);
  __syncthreads();
  // Expert e is hot when fewer than n_hot experts precede it in the order
  // (count descending, id ascending).
  int flags = 0;  // bit q: expert tid * kPerThread + q is hot
  int my_hot = 0;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int e = tid * kPerThread + q;
    if (e >= a.E) break;
    const int c = cnt[e];
    int rank = 0;
    for (int f = 0; f < a.E; ++f) {
      const int cf = cnt[f];
      rank += (cf > c || (cf == c && f < e)) ? 1 : 0;
    }
    if (rank < a.n_hot) {
      flags |= 1 << q;
      ++my_hot;
    }
  }
  // Exclusive prefix of the hot flags over threads (ids ascending).
  const int incl = warp_inclusive_sum(my_hot, lane);
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int t = warp_inclusive_sum(warp_tot[lane], lane);
    warp_tot[lane] = t;
  }
  __syncthreads();
  int pos = incl - my_hot + (wid > 0 ? warp_tot[wid - 1] : 0);
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int e = tid * kPerThread + q;
    if (e >= a.E) break;
    const bool h = (flags >> q) & 1;
    if (a.counts) a.counts[e] = cnt[e];
    if (h) a.hot[pos] = e;
    if (a.home_slot) a.home_slot[e] = h ? a.first_slot + pos : -1;
    pos += h ? 1 : 0;
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_hot_list(const int32_t* ids, int64_t n_ids, int32_t E, int32_t n_hot, int32_t first_slot,
                            int32_t* counts, int32_t* hot, int32_t* home_slot, int32_t* dev_err, void* stream) {
  using namespace moe;
  if (E < 1 || E > kHotMaxE || n_hot < 0 || n_hot > E || n_ids < 0 || n_ids > INT32_MAX) return MOE_ERR_ARG;
  if (first_slot < 0 || static_cast<long long>(first_slot) + n_hot > INT32_MAX) return MOE_ERR_ARG;
  if ((n_ids > 0 && !ids) || (n_hot > 0 && !hot)) return MOE_ERR_ARG;
  HotArgs a{ids, static_cast<long long>(n_ids), E, n_hot, first_slot, counts, hot, home_slot, dev_err};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope ls(kProfHot, s);
  return launch_k(hot_list_kernel, dim3(1), dim3(kHotThreads), 0, s, false, a);
}
