// Device-side expert union / permutation shared by moe_union_permute and the
// fused layer-head kernel.
//
// EcoSpec write-up, section 2: the experts a verify step loads in a layer are
// the union of the experts its tokens route to.  S2-MoE write-up, challenge 2:
// reuse ratio |union| / (s * k).  A token x expert membership bitmap in shared
// memory (atomicOr, which also catches duplicate ids) gives the union (one warp
// scans <= 1024 experts in ascending order) and each pair's rank in its expert
// group (popcount of the expert's column over earlier tokens): a deterministic
// permutation without a sort.
#pragma once

#include "common.cuh"

namespace moe {
namespace unions {

constexpr int kMaxE = 1024;

struct UnionSmem {
  int32_t count[kMaxE];
  int32_t ustart[kMaxE];  // expert -> first perm position of its group
  int err;
};

struct UnionView {
  int32_t* count;   // [E]
  int32_t* ustart;  // [E]
  int* err;
};

__device__ __forceinline__ UnionView view_of(UnionSmem& us) { return UnionView{us.count, us.ustart, &us.err}; }

__host__ __device__ inline size_t union_view_bytes(int E) { return 4 * (2 * static_cast<size_t>(E) + 1); }

__device__ __forceinline__ UnionView carve_union(uint8_t* p, int E) {
  UnionView v;
  v.count = reinterpret_cast<int32_t*>(p);
  v.ustart = v.count + E;
  v.err = v.ustart + E;
  return v;
}

// All threads of the block must call it; `member` holds T * ceil(E/32) words.
__device__ __forceinline__ void union_block(const int32_t* __restrict__ ids, int T, int k, int E, uint32_t* member, UnionView us,
                            int32_t* __restrict__ n_unique, int32_t* __restrict__ unique,
                            int32_t* __restrict__ offsets, int32_t* __restrict__ perm_token,
                            int32_t* __restrict__ perm_slot, int32_t* __restrict__ inv,
                            float* __restrict__ reuse_ratio, int32_t* dev_err) {
  const int EW = (E + 31) >> 5;
  const int TK = T * k;
  for (int i = threadIdx.x; i < T * EW; i += blockDim.x) member[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) us.count[e] = 0;
  if (threadIdx.x == 0) *us.err = 0;
  __syncthreads();

  for (int p = threadIdx.x; p < TK; p += blockDim.x) {
    int t = p / k;
    int e = ids[p];
    if (e < 0 || e >= E) {
      atomicOr(us.err, MOE_DEV_BAD_ID);
      continue;
    }
    uint32_t bit = 1u << (e & 31);
    uint32_t old = atomicOr(&member[t * EW + (e >> 5)], bit);
    if (old & bit) atomicOr(us.err, MOE_DEV_DUP_ID);
    atomicAdd(&us.count[e], 1);
  }
  __syncthreads();
  const int err = *us.err;
  if (err) {
    if (threadIdx.x == 0) {
      flag_error(dev_err, err);
      *n_unique = 0;
      *reuse_ratio = 0.f;
      offsets[0] = 0;
    }
    return;
  }

  // Union + group starts: warp 0 scans experts in ascending order.
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int nz = 0, tok = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) {
      nz += us.count[e] > 0;
      tok += us.count[e];
    }
    int nz_ex = nz, tok_ex = tok;  // inclusive -> exclusive scan
    warp_inclusive_sum2(nz_ex, tok_ex, lane);
    nz_ex -= nz;
    tok_ex -= tok;
    for (int e = e0; e < e0 + per && e < E; ++e) {
      if (us.count[e] > 0) {
        us.ustart[e] = tok_ex;
        unique[nz_ex] = e;
        offsets[nz_ex] = tok_ex;
        ++nz_ex;
        tok_ex += us.count[e];
      }
    }
    if (lane == 31) {
      offsets[nz_ex] = tok_ex;  // == T*k
      *n_unique = nz_ex;
      *reuse_ratio = TK > 0 ? __fdiv_rn(static_cast<float>(nz_ex), static_cast<float>(TK)) : 0.f;
    }
  }
  __syncthreads();

  // Permutation: rank of token t in expert e's group = set bits of column e
  // over tokens t' < t.
  for (int p = threadIdx.x; p < TK; p += blockDim.x) {
    int t = p / k;
    int j = p - t * k;
    int e = ids[p];
    int word = e >> 5;
    uint32_t bit = 1u << (e & 31);
    int rank = 0;
    for (int tt = 0; tt < t; ++tt) rank += (member[tt * EW + word] & bit) ? 1 : 0;
    int pos = us.ustart[e] + rank;
    perm_token[pos] = t;
    perm_slot[pos] = j;
    inv[p] = pos;
  }
}

}  // namespace unions
}  // namespace moe
