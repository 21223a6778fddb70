// moe_route: router top-k + softmax weights, with the optional S2-MoE
// reuse-aware soft bias.
//
// Routing follows the EcoSpec write-up, section 3.1 (softmax over the gate
// logits, top-K per layer); the bias follows the S2-MoE write-up, component 2
// (reuse-aware expert gating, steps 1-3 and Fig. 5): a confidence-weighted
// expert importance g_e, a bounded preferred set E* of the top `cap` experts,
// and an additive per-token bias lambda_b proportional to the margin between
// the token's top-1 and (k+1)-th logits.
//
// Design: one warp owns one token; each lane holds ceil(E/32) logits in
// registers and the top-k is k rounds of a warp-wide arg-max (butterfly
// shuffles over a strict total order: larger value, then lower id).  The
// biased variant runs in a single CTA because g_e aggregates over all tokens.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxK = 16;

template <int NPL>
struct Row {
  float v[NPL];
  uint32_t taken;
};

// Loads one logits row; with `estar` set, adds lam to the preferred experts
// (fp32 add, no contraction).  Returns true if any value is NaN.
template <int NPL>
__device__ __forceinline__ bool load_row(const float* __restrict__ row, int E, int lane, Row<NPL>& r,
                                         const uint32_t* estar, float lam) {
  bool nan = false;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    int e = lane + 32 * j;
    float x = -INFINITY;
    if (e < E) {
      x = row[e];
      nan |= (x != x);
      if (estar && ((estar[e >> 5] >> (e & 31)) & 1u)) x = __fadd_rn(x, lam);
    }
    r.v[j] = x;
  }
  r.taken = 0;
  return __any_sync(kFull, nan);
}

// One arg-max round over the not-yet-taken entries; every lane gets the result.
template <int NPL>
__device__ __forceinline__ void argmax_round(Row<NPL>& r, int E, int lane, float& bv, int& bi) {
  float lv = -INFINITY;
  int li = INT_MAX;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    int e = lane + 32 * j;
    if (e < E && !((r.taken >> j) & 1u) && topk_better(r.v[j], e, lv, li)) {
      lv = r.v[j];
      li = e;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(kFull, lv, off);
    int oi = __shfl_xor_sync(kFull, li, off);
    if (topk_better(ov, oi, lv, li)) {
      lv = ov;
      li = oi;
    }
  }
  if (li != INT_MAX && (li & 31) == lane) r.taken |= 1u << (li >> 5);
  bv = lv;
  bi = li;
}

// Top-k of a loaded row and softmax over the selected logits; writes the
// token's ids and weights.  The weight sum runs over j = 0..k-1 in order.
template <int NPL>
__device__ __forceinline__ void topk_softmax_write(Row<NPL>& r, int E, int k, int lane, int32_t* ids,
                                                   float* w) {
  float sv[kMaxK];
  int si[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) argmax_round(r, E, lane, sv[j], si[j]);
  }
  const float m = sv[0];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k) s = __fadd_rn(s, expf(sv[j] - m));
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k && lane == j) {
      ids[j] = si[j];
      w[j] = __fdiv_rn(expf(sv[j] - m), s);
    }
  }
}

__device__ __forceinline__ void write_invalid(int k, int lane, int32_t* ids, float* w) {
  for (int j = lane; j < k; j += 32) {
    ids[j] = -1;
    w[j] = 0.f;
  }
}

template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits,
                                                    const int32_t* __restrict__ rows, int rows_limit,
                                                    int T, int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w, int32_t* dev_err) {
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp; t < T; t += nwarps) {
    const long long row = rows ? rows[t] : t;
    if (rows && (row < 0 || row >= rows_limit)) {
      if (lane == 0) flag_error(dev_err, MOE_DEV_CAPACITY);
      write_invalid(k, lane, ids + (size_t)t * k, w + (size_t)t * k);
      continue;
    }
    Row<NPL> r;
    bool nan = load_row<NPL>(logits + row * E, E, lane, r, nullptr, 0.f);
    if (nan) {
      if (lane == 0) flag_error(dev_err, MOE_DEV_NAN_LOGIT);
      write_invalid(k, lane, ids + (size_t)t * k, w + (size_t)t * k);
      continue;
    }
    topk_softmax_write<NPL>(r, E, k, lane, ids + (size_t)t * k, w + (size_t)t * k);
  }
}

// Single-CTA biased routing (S2-MoE component 2).  T <= 256, E <= 1024;
// 8 warps loop over the tokens.
template <int NPL>
__global__ void __launch_bounds__(256) route_bias_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ rows, int rows_limit,
    const float* __restrict__ w_conf, int T, int E, int k, int cap, float alpha,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* dev_err) {
  constexpr int kMaxT = 256;
  constexpr int kEW = 32;  // 1024 experts / 32
  __shared__ uint32_t member[kMaxT][kEW];
  __shared__ float v1[kMaxT], vk1[kMaxT];
  __shared__ uint8_t bad[kMaxT];
  __shared__ float g[1024];
  __shared__ uint32_t estar[kEW];
  __shared__ int conf_bad;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int EW = (E + 31) >> 5;

  if (threadIdx.x == 0) conf_bad = 0;
  for (int i = threadIdx.x; i < kEW; i += blockDim.x) estar[i] = 0;
  __syncthreads();
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    float c = w_conf[t];
    if (!(c >= 0.f)) conf_bad = 1;  // NaN or negative
  }
  // Pass 1: original top-(k+1) per token -> membership of TopK, l_(1), l_(k+1).
  for (int t = warp; t < T; t += nwarps) {
    const long long row = rows ? rows[t] : t;
    for (int i = lane; i < EW; i += 32) member[t][i] = 0;
    if (rows && (row < 0 || row >= rows_limit)) {
      if (lane == 0) bad[t] = 2;
      continue;
    }
    Row<NPL> r;
    bool nan = load_row<NPL>(logits + row * E, E, lane, r, nullptr, 0.f);
    if (lane == 0) bad[t] = nan ? 1 : 0;
    if (nan) continue;
    __syncwarp();
    for (int j = 0; j <= k; ++j) {
      float bv;
      int bi;
      argmax_round(r, E, lane, bv, bi);
      if (lane == 0) {
        if (j == 0) v1[t] = bv;
        if (j == k) vk1[t] = bv;
        if (j < k) member[t][bi >> 5] |= 1u << (bi & 31);
      }
    }
  }
  __syncthreads();
  if (conf_bad) {
    if (threadIdx.x == 0) flag_error(dev_err, MOE_DEV_BAD_PROB);
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
      ids[i] = -1;
      w[i] = 0.f;
    }
    return;
  }
  // Step 1: g_e = sum over tokens (ascending) of w_b for tokens whose top-k holds e.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
    for (int b = 0; b < T; ++b)
      if (!bad[b] && ((member[b][e >> 5] >> (e & 31)) & 1u)) acc = __fadd_rn(acc, w_conf[b]);
    g[e] = acc;
  }
  __syncthreads();
  // Step 2: E* = top-cap experts by g among g > 0 (ties: lower id).
  if (warp == 0) {
    uint32_t taken = 0;  // bit j: expert lane + 32 j
    for (int c = 0; c < cap; ++c) {
      float lv = -INFINITY;
      int li = INT_MAX;
      for (int j = 0; j < EW; ++j) {
        int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && g[e] > 0.f && topk_better(g[e], e, lv, li)) {
          lv = g[e];
          li = e;
        }
      }
      for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(kFull, lv, off);
        int oi = __shfl_xor_sync(kFull, li, off);
        if (topk_better(ov, oi, lv, li)) {
          lv = ov;
          li = oi;
        }
      }
      if (li == INT_MAX) break;  // no expert left with g > 0
      if ((li & 31) == lane) taken |= 1u << (li >> 5);
      if (lane == 0) estar[li >> 5] |= 1u << (li & 31);
    }
  }
  __syncthreads();
  // Step 3 + routing on the biased logits.
  for (int t = warp; t < T; t += nwarps) {
    int32_t* ti = ids + (size_t)t * k;
    float* tw = w + (size_t)t * k;
    if (bad[t]) {
      if (lane == 0) flag_error(dev_err, bad[t] == 2 ? MOE_DEV_CAPACITY : MOE_DEV_NAN_LOGIT);
      write_invalid(k, lane, ti, tw);
      continue;
    }
    const float lam = __fmul_rn(alpha, __fsub_rn(v1[t], vk1[t]));
    const long long row = rows ? rows[t] : t;
    Row<NPL> r;
    load_row<NPL>(logits + row * E, E, lane, r, estar, lam);
    topk_softmax_write<NPL>(r, E, k, lane, ti, tw);
  }
}

template <int NPL>
int launch_npl(const RouteArgs& a) {
  const auto& c = a.cfg;
  if (c.use_bias) {
    int threads = 32 * (c.T < 8 ? (c.T < 1 ? 1 : c.T) : 8);
    LaunchScope ls(kProfRoute, a.stream);
    route_bias_kernel<NPL><<<1, threads, 0, a.stream>>>(a.logits, a.rows, a.rows_limit, a.w_conf,
                                                         c.T, c.E, c.k, c.cap, c.alpha, a.ids, a.w,
                                                         a.dev_err);
  } else {
    int warps = c.T;
    int blocks = (warps + 7) / 8;
    LaunchScope ls(kProfRoute, a.stream);
    route_kernel<NPL><<<blocks, 256, 0, a.stream>>>(a.logits, a.rows, a.rows_limit, c.T, c.E, c.k,
                                                    a.ids, a.w, a.dev_err);
  }
  return check_launch();
}

}  // namespace

int route_validate(const moe_route_cfg& c, bool have_conf) {
  if (c.T < 0 || c.k < 1 || c.k > kMaxK || c.E < c.k || c.E > 1024) return MOE_ERR_UNSUPPORTED;
  if (c.use_bias) {
    if (!have_conf || c.cap < 1 || c.E < c.k + 1) return MOE_ERR_ARG;
    if (c.T > 256) return MOE_ERR_UNSUPPORTED;
    if (!(c.alpha == c.alpha)) return MOE_ERR_ARG;
  }
  return MOE_OK;
}

int route_launch(const RouteArgs& a) {
  if (a.cfg.T == 0) return MOE_OK;
  int npl = (a.cfg.E + 31) / 32;
  if (npl <= 1) return launch_npl<1>(a);
  if (npl <= 2) return launch_npl<2>(a);
  if (npl <= 4) return launch_npl<4>(a);
  if (npl <= 8) return launch_npl<8>(a);
  if (npl <= 16) return launch_npl<16>(a);
  return launch_npl<32>(a);
}

}  // namespace moe

extern "C" int moe_route(const float* logits, const float* w_conf, const moe_route_cfg* cfg,
                         int32_t* ids, float* w, int32_t* dev_err, void* stream) {
  if (!cfg) return MOE_ERR_ARG;
  int st = moe::route_validate(*cfg, w_conf != nullptr);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!logits || !ids || !w)) return MOE_ERR_ARG;
  moe::RouteArgs a{logits, nullptr, 0, w_conf, *cfg, ids, w, dev_err, static_cast<cudaStream_t>(stream)};
  return moe::route_launch(a);
}
