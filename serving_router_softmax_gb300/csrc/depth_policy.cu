// moe_depth_policy: the confidence-gated depth vector of ragged speculation.
//
// Width-vs-depth note, section 2: every step, choose one speculation depth
// per live sequence so that the expected batch throughput is largest; first
// a batch-common depth from the live sequences' confidences, then greedy
// truncation of single sequences while that raises the expected throughput.
// The draft's confidence at depth j is the cumulative product of its
// per-token confidences (calibrated against the committed length).
//
// Readings (the oracle applies the same ones):
//   A_i(d)   = 1 + c_i1 + ... + c_id            expected committed tokens
//   cost(d)  = C0 + T_exp * U(d)                U = distinct (layer, expert)
//              pairs over the predicted footprints of every verified position
//              (each root, position 0, always)
//   thr(d)   = sum_i A_i(d_i) / cost(d)
// common depth: d_i = min(D', max_i), best D' (ties to the smaller D');
// truncation: repeatedly the single decrement with the largest thr, if
// strictly larger (ties to the lower sequence).  fp64 with a fixed order and
// no contraction: A_i(j) = A_i(j-1) + c_ij; num summed over i ascending from
// 0; den = C0 + (T_exp * U); thr = num / den.
//
// One CTA.  The footprints become per-sequence prefix unions in shared
// memory, union sizes are integer popcounts (exact whatever the order of the
// atomics); in a truncation round every candidate's union comes from one
// pass: the union of the current vector, the bits covered by two or more
// sequences, and per candidate the bits only its last position adds.
#include <cmath>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kDepthThreads = 256;
constexpr int kDepthMaxSeq = kDepthThreads;   // one candidate per thread
constexpr int kDepthMaxD = 32;
constexpr size_t kDepthMaxSmem = 200 * 1024;

struct DepthArgs {
  const float* conf;
  const uint32_t* fp;
  const int32_t* max_depth;
  int nseq, D, W;
  double C0, T_exp;
  int32_t* depth;
  int32_t* common;
  double* thr;
  int32_t* dev_err;
};

size_t depth_smem_bytes(int nseq, int D, int W) {
  return static_cast<size_t>(nseq) * (D + 1) * sizeof(double)            // A
         + static_cast<size_t>(nseq) * (D + 1) * W * sizeof(uint32_t);   // prefix unions
}

__device__ __forceinline__ double thr_of(double num, double C0, double T_exp, int U) {
  return __ddiv_rn(num, __dadd_rn(C0, __dmul_rn(T_exp, static_cast<double>(U))));
}

// (value, index) arg-max over the block: larger value wins, equal values go
// to the lower index; index -1 means no candidate.
__device__ void block_argmax(double v, int idx, double* sv, int* si, double* out_v, int* out_i) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double ov = __shfl_down_sync(0xFFFFFFFFu, v, off);
    const int oi = __shfl_down_sync(0xFFFFFFFFu, idx, off);
    if (oi >= 0 && (idx < 0 || ov > v || (ov == v && oi < idx))) {
      v = ov;
      idx = oi;
    }
  }
  if (lane == 0) {
    sv[wid] = v;
    si[wid] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double bv = 0.0;
    int bi = -1;
    for (int w = 0; w < kDepthThreads / 32; ++w) {
      if (si[w] >= 0 && (bi < 0 || sv[w] > bv || (sv[w] == bv && si[w] < bi))) {
        bv = sv[w];
        bi = si[w];
      }
    }
    *out_v = bv;
    *out_i = bi;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDepthThreads) depth_policy_kernel(const DepthArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int nseq = a.nseq, D = a.D, W = a.W, D1 = D + 1;
  double* A = reinterpret_cast<double*>(smem);                              // [nseq][D+1]
  uint32_t* pre = reinterpret_cast<uint32_t*>(A + static_cast<size_t>(nseq) * D1);  // [nseq][D+1][W]
  __shared__ int d[kDepthMaxSeq];
  __shared__ int lim[kDepthMaxSeq];
  __shared__ int lost[kDepthMaxSeq];
  __shared__ int cnt[kDepthMaxD + 1];
  __shared__ int u_full;
  __shared__ int bad;
  __shared__ double red_v[kDepthThreads / 32];
  __shared__ int red_i[kDepthThreads / 32];
  __shared__ double best_v;
  __shared__ int best_i;
  __shared__ int best_D;
  __shared__ double cur;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();

  if (tid == 0) {
    bad = 0;
    u_full = 0;
  }
  for (int j = tid; j <= D; j += kDepthThreads) cnt[j] = 0;
  // Prefix unions of the footprints: pre[i][j] = OR of positions 0..j.
  for (int p = tid; p < nseq * W; p += kDepthThreads) {
    const int i = p / W, w = p - i * W;
    uint32_t acc = 0;
    for (int j = 0; j < D1; ++j) {
      const size_t o = (static_cast<size_t>(i) * D1 + j) * W + w;
      acc |= a.fp[o];
      pre[o] = acc;
    }
  }
  __syncthreads();
  // Expected committed tokens per depth, fp64 in depth order.
  if (tid < nseq) {
    double acc = 1.0;
    A[tid * D1] = acc;
    bool ok = true;
    for (int j = 0; j < D; ++j) {
      const float c = a.conf[static_cast<size_t>(tid) * D + j];
      ok = ok && c >= 0.f && c <= 1.f;  // false for NaN
      acc = __dadd_rn(acc, static_cast<double>(c));
      A[tid * D1 + j + 1] = acc;
    }
    if (!ok) atomicOr(&bad, 1);
    int m = a.max_depth ? a.max_depth[tid] : D;
    lim[tid] = m < 0 ? 0 : (m > D ? D : m);
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      flag_error(a.dev_err, MOE_DEV_BAD_PROB);
      if (a.common) *a.common = 0;
      if (a.thr) a.thr[0] = a.thr[1] = 0.0;
    }
    for (int i = tid; i < nseq; i += kDepthThreads) a.depth[i] = 0;
    return;
  }

  // ---- batch-common depth: union size for every D' in one pass.
  for (int p = tid; p < D1 * W; p += kDepthThreads) {
    const int Dc = p / W, w = p - Dc * W;
    uint32_t u = 0;
    for (int i = 0; i < nseq; ++i) {
      const int di = Dc < lim[i] ? Dc : lim[i];
      u |= pre[(static_cast<size_t>(i) * D1 + di) * W + w];
    }
    if (u) atomicAdd(&cnt[Dc], __popc(u));
  }
  __syncthreads();
  if (tid == 0) {
    double bv = 0.0;
    int bD = -1;
    for (int Dc = 0; Dc <= D; ++Dc) {
      double num = 0.0;
      for (int i = 0; i < nseq; ++i) num = __dadd_rn(num, A[i * D1 + (Dc < lim[i] ? Dc : lim[i])]);
      const double t = thr_of(num, a.C0, a.T_exp, cnt[Dc]);
      if (bD < 0 || t > bv) {
        bv = t;
        bD = Dc;
      }
    }
    best_D = bD;
    cur = bv;
    if (a.thr) a.thr[0] = bv;
    if (a.common) *a.common = bD;
  }
  __syncthreads();
  for (int i = tid; i < nseq; i += kDepthThreads) d[i] = best_D < lim[i] ? best_D : lim[i];
  __syncthreads();

  // ---- greedy truncation.
  for (int round = 0; round <= nseq * D; ++round) {
    for (int i = tid; i < nseq; i += kDepthThreads) lost[i] = 0;
    if (tid == 0) u_full = 0;
    __syncthreads();
    for (int w = tid; w < W; w += kDepthThreads) {
      uint32_t once = 0, twice = 0;
      for (int i = 0; i < nseq; ++i) {
        const uint32_t c = pre[(static_cast<size_t>(i) * D1 + d[i]) * W + w];
        twice |= once & c;
        once |= c;
      }
      if (once) atomicAdd(&u_full, __popc(once));
      for (int i = 0; i < nseq; ++i) {
        if (d[i] == 0) continue;
        const uint32_t top = pre[(static_cast<size_t>(i) * D1 + d[i]) * W + w];
        const uint32_t below = pre[(static_cast<size_t>(i) * D1 + d[i] - 1) * W + w];
        const uint32_t gone = top & ~below & ~twice;
        if (gone) atomicAdd(&lost[i], __popc(gone));
      }
    }
    __syncthreads();
    double v = 0.0;
    int idx = -1;
    if (tid < nseq && d[tid] > 0) {
      double num = 0.0;
      for (int i = 0; i < nseq; ++i) num = __dadd_rn(num, A[i * D1 + d[i] - (i == tid ? 1 : 0)]);
      v = thr_of(num, a.C0, a.T_exp, u_full - lost[tid]);
      idx = tid;
    }
    block_argmax(v, idx, red_v, red_i, &best_v, &best_i);
    const bool take = best_i >= 0 && best_v > cur;
    __syncthreads();
    if (!take) break;
    if (tid == 0) {
      d[best_i] -= 1;
      cur = best_v;
    }
    __syncthreads();
  }
  for (int i = tid; i < nseq; i += kDepthThreads) a.depth[i] = d[i];
  if (tid == 0 && a.thr) a.thr[1] = cur;
}

}  // namespace
}  // namespace moe

extern "C" int moe_depth_policy(const float* conf, const uint32_t* fp, const int32_t* max_depth,
                                const moe_depth_cfg* cfg, int32_t* depth, int32_t* common_depth,
                                double* throughput, int32_t* dev_err, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_ARG;
  const moe_depth_cfg c = *cfg;
  if (c.nseq < 1 || c.nseq > kDepthMaxSeq || c.D < 1 || c.D > kDepthMaxD || c.W < 1) return MOE_ERR_UNSUPPORTED;
  if (!std::isfinite(c.C0) || !(c.C0 > 0.f) || !std::isfinite(c.T_exp) || !(c.T_exp >= 0.f)) return MOE_ERR_ARG;
  const size_t smem = depth_smem_bytes(c.nseq, c.D, c.W);
  if (smem > kDepthMaxSmem) return MOE_ERR_UNSUPPORTED;
  if (!conf || !fp || !depth) return MOE_ERR_ARG;
  DepthArgs a{conf, fp, max_depth, c.nseq, c.D, c.W, static_cast<double>(c.C0), static_cast<double>(c.T_exp),
              depth, common_depth, throughput, dev_err};
  if (cudaFuncSetAttribute(depth_policy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope ls(kProfDepth, s);
  return launch_k(depth_policy_kernel, dim3(1), dim3(kDepthThreads), smem, s, false, a);
}
