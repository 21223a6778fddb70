// s2_expand: S2-MoE routing-aware adaptive speculative expansion.
//
// S2-MoE write-up, component 1: adding draft token i to the selected set S
// costs |E_i \ union_{j in S} E_j| * T_exp (new experts the target must load)
// plus C_draft; its utility is p_i * T_AR over that cost; candidates are taken
// while their utility is at least 1, until none qualifies.
//
// A node is a candidate once its parent is selected (children of the root
// always are), which keeps the selection prefix-closed.  Taking a node only
// lowers the other nodes' costs and only adds candidates, so the selected set
// is the least fixed point of a monotone rule: it does not depend on the order
// in which candidates are examined.  The kernel therefore evaluates every
// candidate of a round against the same union in parallel (one warp per node,
// popcounts of E_i & ~B over the bitset words) and takes all that qualify, then
// repeats; the page's one-by-one pass in draft order reaches the same set.
// U_i >= 1 is evaluated as p_i * T_AR >= n_new * T_exp + C_draft in fp64 with
// that operation order (both products exact, the addition rounded once).
//
// Expert residency: the write-up prices an expert by its bytes over the
// bandwidth it is moved at.  With a mask of non-resident experts, a new expert
// that is also cold costs T_cold more (it crosses the host link before HBM):
// cost = (n_new * T_exp + n_new_cold * T_cold) + C_draft.
//
// One CTA per sequence; footprints live in shared memory as bitsets.
#include <cmath>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kS2MaxN = 1024;
constexpr int kS2MaxW = 4096;
constexpr int kS2MaxNW = 40960;  // N*W words of footprint bitsets (160 KB)

__global__ void __launch_bounds__(512) s2_kernel(const float* __restrict__ P, const int32_t* __restrict__ parent,
                                                 const uint32_t* __restrict__ own_fp, int N, int W, double t_ar,
                                                 double t_exp, double c_draft, double t_cold,
                                                 const uint32_t* __restrict__ cold_fp, int32_t* __restrict__ selected,
                                                 int32_t* __restrict__ n_selected, int32_t* __restrict__ union_size,
                                                 int32_t* dev_err) {
  extern __shared__ uint32_t smem[];
  uint32_t* fp = smem;               // [N][W] own footprints
  uint32_t* B = fp + (size_t)N * W;  // [W] union of the selected footprints
  uint32_t* cold = B + W;            // [W] non-resident experts (when cold_fp is given)
  __shared__ uint8_t chosen[kS2MaxN];
  __shared__ uint8_t take[kS2MaxN];
  __shared__ int16_t par_s[kS2MaxN];
  __shared__ int bad;

  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const float* Ps = P + (size_t)s * N;
  const int32_t* par = parent + (size_t)s * N;
  const uint32_t* own = own_fp + (size_t)s * N * W;
  int32_t* sel = selected + (size_t)s * N;

  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int t = threadIdx.x; t < N; t += blockDim.x) {
    const int p = par[t];
    if (p < -1 || p >= t) atomicOr(&bad, MOE_DEV_BAD_TREE);
    const float pt = Ps[t];
    if (!(pt >= 0.f) || pt == INFINITY) atomicOr(&bad, MOE_DEV_BAD_PROB);
    par_s[t] = static_cast<int16_t>(p);
    chosen[t] = 0;
  }
  for (int i = threadIdx.x; i < N * W; i += blockDim.x) fp[i] = own[i];
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    B[w] = 0;
    cold[w] = cold_fp ? cold_fp[w] : 0u;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      flag_error(dev_err, bad);
      n_selected[s] = 0;
      union_size[s] = 0;
    }
    for (int t = threadIdx.x; t < N; t += blockDim.x) sel[t] = -1;
    return;
  }

  // Rounds: every candidate against the current union; take all that
  // qualify.  Each round that continues takes at least one node.
  for (int round = 0; round <= N; ++round) {
    for (int t = warp; t < N; t += nwarps) {
      const bool cand = !chosen[t] && (par_s[t] < 0 || chosen[par_s[t]]);
      int c = 0, cc = 0;
      if (cand) {
        const uint32_t* ft = fp + (size_t)t * W;
        for (int w = lane; w < W; w += 32) {
          const uint32_t nw = ft[w] & ~B[w];
          c += __popc(nw);
          cc += __popc(nw & cold[w]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
          cc += __shfl_xor_sync(0xFFFFFFFFu, cc, off);
        }
      }
      if (lane == 0) {
        bool tk = false;
        if (cand) {
          const double gain = __dmul_rn(static_cast<double>(Ps[t]), t_ar);
          const double moved = __dadd_rn(__dmul_rn(static_cast<double>(c), t_exp),
                                         __dmul_rn(static_cast<double>(cc), t_cold));
          const double cost = __dadd_rn(moved, c_draft);
          tk = gain >= cost;
        }
        take[t] = tk ? 1 : 0;
      }
    }
    __syncthreads();
    int any = 0;
    for (int t = threadIdx.x; t < N; t += blockDim.x)
      if (take[t]) {
        chosen[t] = 1;
        any = 1;
      }
    for (int w = threadIdx.x; w < W; w += blockDim.x) {
      uint32_t add = 0;
      for (int t = 0; t < N; ++t)
        if (take[t]) add |= fp[(size_t)t * W + w];
      B[w] |= add;
    }
    if (!__syncthreads_or(any)) break;
  }

  // Selected nodes in ascending order, then -1; count and |union|.
  if (warp == 0) {
    int base = 0;
    for (int t0 = 0; t0 < N; t0 += 32) {
      const int t = t0 + lane;
      const bool on = t < N && chosen[t];
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, on);
      if (on) sel[base + __popc(m & ((1u << lane) - 1u))] = t;
      base += __popc(m);
    }
    for (int q = base + lane; q < N; q += 32) sel[q] = -1;
    int c = 0;
    for (int w = lane; w < W; w += 32) c += __popc(B[w]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    if (lane == 0) {
      n_selected[s] = base;
      union_size[s] = c;
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" int s2_expand(const float* P, const int32_t* parent, const uint32_t* own_fp, int32_t nseq,
                         const s2_cfg* cfg, int32_t* selected, int32_t* n_selected, int32_t* union_size,
                         int32_t* dev_err, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_ARG;
  const s2_cfg& c = *cfg;
  if (nseq < 0) return MOE_ERR_ARG;
  if (c.N < 1 || c.N > kS2MaxN || c.W < 1 || c.W > kS2MaxW ||
      static_cast<long long>(c.N) * c.W > kS2MaxNW)
    return MOE_ERR_UNSUPPORTED;
  if (!std::isfinite(c.T_AR) || !std::isfinite(c.T_exp) || !std::isfinite(c.C_draft) || !std::isfinite(c.T_cold) ||
      c.T_AR < 0.f || c.T_exp < 0.f || c.C_draft < 0.f || c.T_cold < 0.f)
    return MOE_ERR_ARG;
  if (nseq == 0) return MOE_OK;
  if (!P || !parent || !own_fp || !selected || !n_selected || !union_size) return MOE_ERR_ARG;
  const size_t smem = (static_cast<size_t>(c.N) * c.W + 2 * static_cast<size_t>(c.W)) * sizeof(uint32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(s2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  const int threads = c.W >= 256 || c.N >= 16 ? 512 : 256;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope ls(kProfS2, s);
  s2_kernel<<<nseq, threads, smem, s>>>(P, parent, own_fp, c.N, c.W, static_cast<double>(c.T_AR),
                                        static_cast<double>(c.T_exp), static_cast<double>(c.C_draft),
                                        static_cast<double>(c.T_cold), c.cold_fp, selected, n_selected, union_size,
                                        dev_err);
  return check_launch();
}
