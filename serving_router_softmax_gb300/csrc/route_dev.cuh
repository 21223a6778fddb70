// Device-side routing building blocks shared by the moe_route kernels and the
// fused layer-head kernel of the whole step.
//
// Routing: EcoSpec write-up, section 3.1 (softmax over the gate logits, top-K
// per layer).  Reuse bias: S2-MoE write-up, component 2 (steps 1-3, Fig. 5).
// One warp owns one token; each lane keeps ceil(E/32) logits in registers and
// the top-k is k rounds of a warp-wide arg-max over a strict total order
// (larger value, then lower id).  Each round is two warp reductions
// (redux.sync): the largest order key, then the lowest expert id holding it.
#pragma once

#include <cfloat>
#include <climits>

#include "common.cuh"

namespace moe {
namespace routing {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxK = 16;

// Order key of a non-NaN float: a larger value has a larger key, -0.0 and
// +0.0 share one key, and no value maps to 0 (which marks "no entry").
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);  // -0.0 -> +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int NPL>
struct Row {
  uint32_t key[NPL];  // order keys; 0 for entries past E
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
    uint32_t key = 0;
    if (e < E) {
      float x = row[e];
      nan |= (x != x);
      if (estar && ((estar[e >> 5] >> (e & 31)) & 1u)) x = __fadd_rn(x, lam);
      key = order_key(x);
    }
    r.key[j] = key;
  }
  r.taken = 0;
  return __any_sync(kFull, nan);
}

// One arg-max round over the not-yet-taken entries; every lane gets the
// result (bi = INT_MAX when nothing is left).  The lane's own entries are
// scanned in ascending id order with a strict compare, so its candidate is
// its lowest id among its largest keys; across lanes the lowest id among the
// lanes holding the largest key wins.
template <int NPL>
__device__ __forceinline__ void argmax_round(Row<NPL>& r, int E, int lane, float& bv, int& bi) {
  uint32_t lk = 0;
  int li = INT_MAX;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    if (!((r.taken >> j) & 1u) && r.key[j] > lk) {
      lk = r.key[j];
      li = lane + 32 * j;
    }
  }
  const uint32_t mk = __reduce_max_sync(kFull, lk);
  const uint32_t cand = (mk != 0 && lk == mk) ? static_cast<uint32_t>(li) : 0xFFFFFFFFu;
  const uint32_t win = __reduce_min_sync(kFull, cand);
  bi = mk != 0 ? static_cast<int>(win) : INT_MAX;
  bv = mk != 0 ? key_value(mk) : -INFINITY;
  if (bi != INT_MAX && (bi & 31) == lane) r.taken |= 1u << (bi >> 5);
}

// Top-k of a loaded row and softmax over the selected logits; writes the
// token's ids and weights.  Lane j keeps slot j, so the rounds need no
// per-slot arrays; the softmax denominator is a fixed-order warp sum.
template <int NPL>
__device__ __forceinline__ void topk_softmax_write(Row<NPL>& r, int E, int k, int lane, int32_t* ids,
                                                   float* w) {
  float mine_v = -INFINITY, m = 0.f;
  int mine_i = -1;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv;
    int bi;
    argmax_round(r, E, lane, bv, bi);
    if (j == 0) m = bv;
    if (lane == j) {
      mine_v = bv;
      mine_i = bi;
    }
  }
  const float ex = lane < k ? expf(mine_v - m) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
  if (lane < k) {
    ids[lane] = mine_i;
    w[lane] = __fdiv_rn(ex, s);
  }
}

__device__ __forceinline__ void write_invalid(int k, int lane, int32_t* ids, float* w) {
  for (int j = lane; j < k; j += 32) {
    ids[j] = -1;
    w[j] = 0.f;
  }
}

// Plain routing: warps [warp0, warp0 + nwarps) of the grid loop over tokens.
template <int NPL>
__device__ __forceinline__ void route_plain_warps(const float* __restrict__ logits, const int32_t* __restrict__ rows,
                                                  int rows_limit, int T, int E, int k, int32_t* __restrict__ ids,
                                                  float* __restrict__ w, int32_t* dev_err, int warp, int nwarps) {
  const int lane = threadIdx.x & 31;
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

constexpr int kBiasMaxT = 256;
constexpr int kMaxEW = 32;  // 1024 experts / 32

struct BiasSmem {
  uint32_t member[kBiasMaxT * kMaxEW];  // [t][EW] top-k membership bits
  float v1[kBiasMaxT], vk1[kBiasMaxT], wc[kBiasMaxT];
  uint8_t bad[kBiasMaxT];
  float g[1024];
  uint32_t estar[kMaxEW];
  int conf_bad;
};

// Shared-memory working set of the biased routing, as pointers so that it can
// live in a static struct (standalone kernel) or be sized to T and E.
struct BiasView {
  uint32_t* member;  // [T][EW]
  float* v1;         // [T]
  float* vk1;        // [T]
  float* wc;         // [T] confidence weights
  uint8_t* bad;      // [T]
  float* g;          // [E]
  uint32_t* estar;   // [EW]
  int* conf_bad;
};

__device__ __forceinline__ BiasView view_of(BiasSmem& sm) {
  return BiasView{sm.member, sm.v1, sm.vk1, sm.wc, sm.bad, sm.g, sm.estar, &sm.conf_bad};
}

// Bytes of a BiasView carved by carve_bias (4-byte aligned pieces).
__host__ __device__ inline size_t bias_view_bytes(int T, int E) {
  const int EW = (E + 31) / 32;
  const size_t Tb = (static_cast<size_t>(T) + 3) & ~size_t(3);
  return 4 * (static_cast<size_t>(T) * EW + 3 * T + E + EW + 1) + Tb;
}

__device__ __forceinline__ BiasView carve_bias(uint8_t* p, int T, int E) {
  const int EW = (E + 31) / 32;
  BiasView v;
  v.member = reinterpret_cast<uint32_t*>(p);
  v.v1 = reinterpret_cast<float*>(v.member + (size_t)T * EW);
  v.vk1 = v.v1 + T;
  v.wc = v.vk1 + T;
  v.g = v.wc + T;
  v.estar = reinterpret_cast<uint32_t*>(v.g + E);
  v.conf_bad = reinterpret_cast<int*>(v.estar + EW);
  v.bad = reinterpret_cast<uint8_t*>(v.conf_bad + 1);
  return v;
}

// Biased routing over the whole block (T <= 256, E <= 1024).  All threads of
// the block must call it; it synchronises the block.
template <int NPL>
__device__ __forceinline__ void route_bias_block(const float* __restrict__ logits, const int32_t* __restrict__ rows,
                                 int rows_limit, const float* __restrict__ w_conf, int T, int E, int k, int cap,
                                 float alpha, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* dev_err,
                                 BiasView sm) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int EW = (E + 31) >> 5;

  for (int i = threadIdx.x; i < EW; i += blockDim.x) sm.estar[i] = 0;
  int my_bad = 0;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const float c = w_conf[t];
    sm.wc[t] = c;
    if (!(c >= 0.f)) my_bad = 1;  // NaN or negative
  }
  // With at most one token per warp, the warp keeps its token's row in
  // registers from the first pass to the second.
  const bool keep = T <= nwarps;
  Row<NPL> kept;
  kept.taken = 0;
  // Pass 1: original top-(k+1) per token -> membership of TopK, l_(1), l_(k+1).
  for (int t = warp; t < T; t += nwarps) {
    const long long row = rows ? rows[t] : t;
    for (int i = lane; i < EW; i += 32) sm.member[t * EW + i] = 0;
    if (rows && (row < 0 || row >= rows_limit)) {
      if (lane == 0) sm.bad[t] = 2;
      continue;
    }
    Row<NPL> r;
    bool nan = load_row<NPL>(logits + row * E, E, lane, r, nullptr, 0.f);
    if (lane == 0) sm.bad[t] = nan ? 1 : 0;
    if (nan) continue;
    if (keep) kept = r;
    __syncwarp();
    for (int j = 0; j <= k; ++j) {
      float bv;
      int bi;
      argmax_round(r, E, lane, bv, bi);
      if (lane == 0) {
        if (j == 0) sm.v1[t] = bv;
        if (j == k) sm.vk1[t] = bv;
        if (j < k) sm.member[t * EW + (bi >> 5)] |= 1u << (bi & 31);
      }
    }
  }
  const bool conf_bad = __syncthreads_or(my_bad) != 0;
  if (!conf_bad) {
    // Step 1: g_e = sum over tokens (ascending) of w_b for tokens whose top-k holds e.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float acc = 0.f;
      for (int b = 0; b < T; ++b)
        if (!sm.bad[b] && ((sm.member[b * EW + (e >> 5)] >> (e & 31)) & 1u)) acc = __fadd_rn(acc, sm.wc[b]);
      sm.g[e] = acc;
    }
  }
  __syncthreads();
  // Step 2: E* = top-cap experts by g among g > 0 (ties: lower id).
  if (!conf_bad && warp == 0) {
    uint32_t taken = 0;  // bit j: expert lane + 32 j
    for (int c = 0; c < cap; ++c) {
      // largest g > 0 among the untaken experts, ties to the lower id (as argmax_round)
      uint32_t lk = 0;
      int li = INT_MAX;
      for (int j = 0; j < EW; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && sm.g[e] > 0.f) {
          const uint32_t key = order_key(sm.g[e]);
          if (key > lk) {
            lk = key;
            li = e;
          }
        }
      }
      const uint32_t mk = __reduce_max_sync(kFull, lk);
      if (mk == 0) break;  // no expert left with g > 0
      const uint32_t win = __reduce_min_sync(kFull, lk == mk ? static_cast<uint32_t>(li) : 0xFFFFFFFFu);
      if (static_cast<int>(win & 31) == lane) taken |= 1u << (win >> 5);
      if (lane == 0) sm.estar[win >> 5] |= 1u << (win & 31);
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
  // Step 3 + routing on the biased logits.
  for (int t = warp; t < T; t += nwarps) {
    int32_t* ti = ids + (size_t)t * k;
    float* tw = w + (size_t)t * k;
    if (sm.bad[t]) {
      if (lane == 0) flag_error(dev_err, sm.bad[t] == 2 ? MOE_DEV_CAPACITY : MOE_DEV_NAN_LOGIT);
      write_invalid(k, lane, ti, tw);
      continue;
    }
    const float lam = __fmul_rn(alpha, __fsub_rn(sm.v1[t], sm.vk1[t]));
    Row<NPL> r;
    if (keep) {
      // l' = l + lam on E*, from the kept keys (key_value(order_key(x)) == x
      // up to the sign of zero, which no comparison or exponent sees)
      r = kept;
      r.taken = 0;
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E && ((sm.estar[e >> 5] >> (e & 31)) & 1u)) r.key[j] = order_key(__fadd_rn(key_value(r.key[j]), lam));
      }
    } else {
      const long long row = rows ? rows[t] : t;
      load_row<NPL>(logits + row * E, E, lane, r, sm.estar, lam);
    }
    topk_softmax_write<NPL>(r, E, k, lane, ti, tw);
  }
}

}  // namespace routing
}  // namespace moe
