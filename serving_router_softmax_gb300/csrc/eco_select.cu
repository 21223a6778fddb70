// eco_select: EcoSpec cost-aware draft selection.
//
// EcoSpec write-up, section 3.2 (the expert buffer B, rebuilt from the empty
// set in every speculative step) and section 3.3 (score
// S(t) = P(t) / (|E_traj(t) \ B| + eps), greedy: take the arg-max node, add it
// to S and merge its path footprint into B, repeat gamma times).  mode 1 is
// the static-cost ablation of section 4.3 (denominator |E_traj(t)|).
//
// Design: one CTA per sequence.  Path footprints E_traj are built once in
// shared memory as bitsets (parent index < child index, so one in-order pass
// per bitset word suffices); every round each warp popcounts (E_traj(t) & ~B)
// for its nodes, warp 0 takes the exact arg-max and all threads OR the winner
// into B.  Scores are compared exactly by cross-multiplication in integers:
// with eps = 2^-s, P_a / (c_a + eps) > P_b / (c_b + eps) iff
// P_a * X_b > P_b * X_a with X = c * 2^s + 1 < 2^29 (checked on the host), and
// P = m * 2^e with a 24-bit integer m, so each side is an integer below 2^53
// times a power of two.  (GB300's fp64 pipe is narrow: the same comparison in
// fp64 cost about 300 cycles per operation in the arg-max chain.)
//
// mode 2 (batch-global): one CTA over the forest of all sequences' trees, one
// buffer B shared by the batch and one greedy with the budget sum(gamma_i) and
// at most min(gamma_max, N) nodes per sequence; each sequence's depth is an
// outcome of the greedy.  The EcoSpec write-up's batch ablation (section 4.3)
// gives no algorithm; this is the plainest batch form of section 3.3, and it
// turns the confidence gating of the width-vs-depth note into a by-product of
// the score.  Ties go to the lower (sequence, node) index.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxN = 1024;
constexpr int kMaxW = 4096;
constexpr int kMaxNW = 40960;  // N*W words of trajectory bitsets (160 KB)

// A node's score P / (c + 2^-s) as exact integers: P = m * 2^e, X = c * 2^s + 1.
struct Score {
  uint32_t m;  // significand of P (< 2^24)
  int e;       // exponent of P
  uint32_t x;  // c * 2^s + 1 (< 2^29)
  int i;       // node index, -1 for none
};

__device__ __forceinline__ Score make_score(float p, int c, int eps_shift, int i) {
  const uint32_t u = __float_as_uint(p);  // p >= 0 and finite (validated)
  const uint32_t ex = (u >> 23) & 0xFFu, fr = u & 0x7FFFFFu;
  Score sc;
  sc.m = ex ? (fr | 0x800000u) : fr;
  sc.e = ex ? static_cast<int>(ex) - 150 : -149;
  sc.x = (static_cast<uint32_t>(c) << eps_shift) + 1u;
  sc.i = i;
  return sc;
}

// Sign of A * 2^ea - B * 2^eb for A, B < 2^54.
__device__ __forceinline__ int cmp_pow2(uint64_t A, int ea, uint64_t B, int eb) {
  if (A == 0 || B == 0) return static_cast<int>(A != 0) - static_cast<int>(B != 0);
  const int la = 63 - __clzll(static_cast<long long>(A)) + ea;  // position of the leading bit
  const int lb = 63 - __clzll(static_cast<long long>(B)) + eb;
  if (la != lb) return la > lb ? 1 : -1;
  // Equal leading positions: the shift keeps the shifted value at the other's bit length.
  if (ea >= eb)
    A <<= (ea - eb);
  else
    B <<= (eb - ea);
  return A > B ? 1 : (A < B ? -1 : 0);
}

// a beats b: P_a / (c_a + eps) > P_b / (c_b + eps), ties -> lower index.
__device__ __forceinline__ bool score_better(const Score& a, const Score& b) {
  const int c = cmp_pow2(static_cast<uint64_t>(a.m) * b.x, a.e, static_cast<uint64_t>(b.m) * a.x, b.e);
  return c > 0 || (c == 0 && a.i < b.i);
}

__device__ __forceinline__ Score shfl_score(const Score& a, int off) {
  Score o;
  o.m = __shfl_xor_sync(0xFFFFFFFFu, a.m, off);
  o.e = __shfl_xor_sync(0xFFFFFFFFu, a.e, off);
  o.x = __shfl_xor_sync(0xFFFFFFFFu, a.x, off);
  o.i = __shfl_xor_sync(0xFFFFFFFFu, a.i, off);
  return o;
}

__device__ __forceinline__ Score shfl_score_from(const Score& a, int src) {
  Score o;
  o.m = __shfl_sync(0xFFFFFFFFu, a.m, src);
  o.e = __shfl_sync(0xFFFFFFFFu, a.e, src);
  o.x = __shfl_sync(0xFFFFFFFFu, a.x, src);
  o.i = __shfl_sync(0xFFFFFFFFu, a.i, src);
  return o;
}

// E_traj(t) = own(t) | E_traj(parent(t)) over nodes 0..G-1 (parent < child):
// one thread per bitset word walks the nodes in order, so every parent is
// final before its children read it.  No barriers between tree levels.
__device__ __forceinline__ void close_paths(uint32_t* traj, const int16_t* par, int G, int W) {
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    for (int g = 0; g < G; ++g) {
      const int p = par[g];
      if (p >= 0) traj[(size_t)g * W + w] |= traj[(size_t)p * W + w];
    }
  }
}

__global__ void __launch_bounds__(512) eco_kernel(
    const float* __restrict__ P, const int32_t* __restrict__ parent,
    const uint32_t* __restrict__ own_fp, const int32_t* __restrict__ gamma_per_seq, int N, int W,
    int gamma_max, int mode, int eps_shift, int fast_key, int32_t* __restrict__ selected,
    int32_t* __restrict__ union_size, int32_t* dev_err, int32_t* __restrict__ verify_rows,
    float* __restrict__ verify_conf, int T_expected, int nseq, int32_t* ready_flag,
    uint32_t* __restrict__ pred_B) {
  extern __shared__ uint32_t smem[];
  if (ready_flag && blockIdx.x == 0 && threadIdx.x == 0) *ready_flag = 0;
  uint32_t* traj = smem;                 // [N][W]
  uint32_t* B = traj + (size_t)N * W;    // [W]
  __shared__ int32_t cost[kMaxN];
  __shared__ float pf[kMaxN];     // P
  __shared__ uint32_t pm[kMaxN];  // P = pm * 2^pe (exact split of the fp32 value)
  __shared__ int16_t pe[kMaxN];
  __shared__ int bad;
  __shared__ int16_t par_s[kMaxN];

  pdl_trigger();  // the first layer's head may launch while selection runs
  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const float* Ps = P + (size_t)s * N;
  const int32_t* par = parent + (size_t)s * N;
  const uint32_t* own = own_fp + (size_t)s * N * W;
  int32_t* sel = selected + (size_t)s * gamma_max;

  int gamma = gamma_per_seq ? gamma_per_seq[s] : gamma_max;

  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  // One pass: own footprints (the trajectories' start), then validation,
  // parents and the split of P, behind a single barrier.
  for (int i = threadIdx.x; i < N * W; i += blockDim.x) traj[i] = own[i];
  for (int t = threadIdx.x; t < N; t += blockDim.x) {
    int p = par[t];
    if (p < -1 || p >= t) atomicOr(&bad, MOE_DEV_BAD_TREE);
    float pt = Ps[t];
    if (!(pt >= 0.f) || pt == INFINITY) atomicOr(&bad, MOE_DEV_BAD_PROB);
    par_s[t] = static_cast<int16_t>(p < -1 || p >= t ? -1 : p);
    const Score sc = make_score(pt >= 0.f ? pt : 0.f, 0, 0, t);
    pf[t] = pt;
    pm[t] = sc.m;
    pe[t] = static_cast<int16_t>(sc.e);
  }
  if (threadIdx.x == 0 && (gamma < 0 || gamma > gamma_max)) atomicOr(&bad, MOE_DEV_BAD_TREE);
  for (int w = threadIdx.x; w < W; w += blockDim.x) B[w] = 0;
  __syncthreads();

  // Optional verify-token map for the whole step (root + selected per sequence).
  int tok0 = 0;
  if (verify_rows) {
    for (int q = 0; q < s; ++q) {
      int gq = gamma_per_seq ? gamma_per_seq[q] : gamma_max;
      gq = gq < 0 ? 0 : (gq > N ? N : gq);
      tok0 += gq + 1;
    }
  }

  if (bad) {
    if (threadIdx.x == 0) {
      flag_error(dev_err, bad);
      union_size[s] = 0;
    }
    for (int r = threadIdx.x; r < gamma_max; r += blockDim.x) sel[r] = -1;
    if (verify_rows) {
      // Keep the downstream gathers in bounds: every token of this sequence
      // points at its root row.
      int g = gamma < 0 ? 0 : (gamma > N ? N : gamma);
      for (int q = threadIdx.x; q <= g; q += blockDim.x)
        if (tok0 + q < T_expected) {
          verify_rows[tok0 + q] = s * (N + 1);
          verify_conf[tok0 + q] = 1.f;
        }
    }
    return;
  }
  if (gamma > N) gamma = N;

  close_paths(traj, par_s, N, W);
  __syncthreads();

  // Rounds.  Every warp computes the same arg-max from the shared costs, so
  // the winner needs no broadcast barrier: two barriers per round.  Lane l
  // tracks in `taken` (bit j) whether node l + 32 j was chosen; the copies
  // agree across warps.
  //
  // Arg-max: when every X = c * 2^s + 1 is below 2^24 (fast_key, checked on
  // the host) X and P are exact fp32 values, so the correctly rounded quotient
  // key = P / X never decreases as the exact score grows: the winner is among
  // the nodes holding the largest key, which a single warp max finds.  Only a
  // tie in the key needs the exact comparison.
  uint32_t taken = 0;
  for (int r = 0; r < gamma; ++r) {
    // Costs: |E_traj(t) \ B| (marginal) or |E_traj(t)| (static).
    for (int t = warp; t < N; t += nwarps) {
      const bool ch = (__shfl_sync(0xFFFFFFFFu, taken, t & 31) >> (t >> 5)) & 1u;
      int c = 0;
      if (!ch) {
        const uint32_t* tt = traj + (size_t)t * W;
#pragma unroll 4
        for (int w = lane; w < W; w += 32) c += __popc(mode == 0 ? (tt[w] & ~B[w]) : tt[w]);
        c = __reduce_add_sync(0xFFFFFFFFu, c);
      }
      if (lane == 0) cost[t] = c;
    }
    __syncthreads();
    Score best{0u, 0, 1u, -1};
    uint32_t best_key = 0;  // key bits + 1 (0: none); keys are >= +0.0
    for (int t = lane, j = 0; t < N; t += 32, ++j) {
      if ((taken >> j) & 1u) continue;
      Score sc;
      sc.m = pm[t];
      sc.e = pe[t];
      sc.x = (static_cast<uint32_t>(cost[t]) << eps_shift) + 1u;
      sc.i = t;
      if (fast_key) {
        const uint32_t kb = __float_as_uint(__fdiv_rn(pf[t], static_cast<float>(sc.x))) + 1u;
        if (kb > best_key || (kb == best_key && score_better(sc, best))) {
          best = sc;
          best_key = kb;
        }
      } else if (best.i < 0 || score_better(sc, best)) {
        best = sc;
      }
    }
    if (fast_key) {
      const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, best_key);
      uint32_t cand = __ballot_sync(0xFFFFFFFFu, best_key == kmax && best.i >= 0);
      Score b = shfl_score_from(best, __ffs(cand) - 1);
      cand &= cand - 1;
      while (cand) {  // lanes whose keys tie: exact comparison (rare)
        const Score o = shfl_score_from(best, __ffs(cand) - 1);
        if (score_better(o, b)) b = o;
        cand &= cand - 1;
      }
      best = b;
    } else {
      for (int off = 16; off > 0; off >>= 1) {
        const Score o = shfl_score(best, off);
        if (o.i >= 0 && (best.i < 0 || score_better(o, best))) best = o;
      }
    }
    const int bi = best.i;  // >= 0: gamma <= N leaves an unchosen node every round
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (threadIdx.x == 0) sel[r] = bi;
    // B |= E_traj(best); the arg-max above reads no B, so this needs no barrier before it.
    const uint32_t* tb = traj + (size_t)bi * W;
    for (int w = threadIdx.x; w < W; w += blockDim.x) B[w] |= tb[w];
    __syncthreads();
  }

  // |B| and the unused slots.
  if (warp == 0) {
    int c = 0;
    for (int w = lane; w < W; w += 32) c += __popc(B[w]);
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    if (lane == 0) union_size[s] = c;
  }
  if (pred_B)
    for (int w = threadIdx.x; w < W; w += blockDim.x) pred_B[(size_t)s * W + w] = B[w];
  for (int r = gamma + threadIdx.x; r < gamma_max; r += blockDim.x) sel[r] = -1;

  if (verify_rows) {
    // Token tok0 is the root (row s*(N+1)); then the selected nodes in order.
    for (int q = threadIdx.x; q <= gamma; q += blockDim.x) {
      int row = s * (N + 1) + (q == 0 ? 0 : 1 + sel[q - 1]);
      float conf = q == 0 ? 1.f : Ps[sel[q - 1]];
      if (tok0 + q < T_expected) {
        verify_rows[tok0 + q] = row;
        verify_conf[tok0 + q] = conf;
      }
    }
    if (threadIdx.x == 0 && s == nseq - 1 && tok0 + gamma + 1 != T_expected)
      flag_error(dev_err, MOE_DEV_CAPACITY);
  }
}

__global__ void __launch_bounds__(512) eco_batch_kernel(
    const float* __restrict__ P, const int32_t* __restrict__ parent, const uint32_t* __restrict__ own_fp,
    const int32_t* __restrict__ gamma_per_seq, int N, int W, int nseq, int gamma_max, int eps_shift,
    int32_t* __restrict__ selected, int32_t* __restrict__ union_size, int32_t* dev_err,
    int32_t* __restrict__ verify_rows, float* __restrict__ verify_conf, int T_expected, int32_t* ready_flag,
    uint32_t* __restrict__ pred_B) {
  extern __shared__ uint32_t smem[];
  if (ready_flag && threadIdx.x == 0) *ready_flag = 0;
  const int G = nseq * N;
  uint32_t* traj = smem;               // [G][W]
  uint32_t* B = traj + (size_t)G * W;  // [W]
  __shared__ int32_t cost[kMaxN];
  __shared__ uint8_t chosen[kMaxN];
  __shared__ int16_t par_s[kMaxN];     // parent as a global node index (-1: root)
  __shared__ int16_t cnt[kMaxN];       // nodes taken per sequence
  __shared__ int bad, best_g, budget;
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int cap = gamma_max < N ? gamma_max : N;

  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int s = g / N, t = g - s * N;
    const int p = parent[g];
    if (p < -1 || p >= t) atomicOr(&bad, MOE_DEV_BAD_TREE);
    const float pt = P[g];
    if (!(pt >= 0.f) || pt == INFINITY) atomicOr(&bad, MOE_DEV_BAD_PROB);
    par_s[g] = static_cast<int16_t>(p < 0 || p >= t ? -1 : s * N + p);
    chosen[g] = 0;
  }
  for (int i = threadIdx.x; i < G * W; i += blockDim.x) traj[i] = own_fp[i];
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int gs = gamma_per_seq ? gamma_per_seq[s] : gamma_max;
    if (gs < 0 || gs > gamma_max) atomicOr(&bad, MOE_DEV_BAD_TREE);
    cnt[s] = 0;
  }
  for (int w = threadIdx.x; w < W; w += blockDim.x) B[w] = 0;
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) flag_error(dev_err, bad);
    for (int i = threadIdx.x; i < nseq * gamma_max; i += blockDim.x) selected[i] = -1;
    for (int s = threadIdx.x; s < nseq; s += blockDim.x) union_size[s] = 0;
    if (verify_rows) {
      // every token points at its sequence's root row (keeps the gathers in bounds)
      if (threadIdx.x == 0) {
        int tok = 0;
        for (int s = 0; s < nseq && tok < T_expected; ++s) {
          int gs = gamma_per_seq ? gamma_per_seq[s] : gamma_max;
          gs = gs < 0 ? 0 : (gs > N ? N : gs);
          for (int q = 0; q <= gs && tok < T_expected; ++q, ++tok) {
            verify_rows[tok] = s * (N + 1);
            verify_conf[tok] = 1.f;
          }
        }
      }
    }
    return;
  }
  if (threadIdx.x == 0) {
    int b = 0;
    for (int s = 0; s < nseq; ++s) {
      int gs = gamma_per_seq ? gamma_per_seq[s] : gamma_max;
      b += gs < N ? gs : N;
    }
    budget = b;
  }

  // Trajectory footprints over the forest (a parent precedes its children).
  close_paths(traj, par_s, G, W);
  __syncthreads();

  for (int r = 0; r < budget; ++r) {
    for (int g = warp; g < G; g += nwarps) {
      int c = 0;
      if (!chosen[g] && cnt[g / N] < cap) {
        const uint32_t* tt = traj + (size_t)g * W;
        for (int w = lane; w < W; w += 32) c += __popc(tt[w] & ~B[w]);
        for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
      }
      if (lane == 0) cost[g] = c;
    }
    __syncthreads();
    if (warp == 0) {
      Score best{0u, 0, 1u, -1};
      for (int g = lane; g < G; g += 32) {
        if (chosen[g] || cnt[g / N] >= cap) continue;
        const Score sc = make_score(P[g], cost[g], eps_shift, g);
        if (best.i < 0 || score_better(sc, best)) best = sc;
      }
      for (int off = 16; off > 0; off >>= 1) {
        const Score o = shfl_score(best, off);
        if (o.i >= 0 && (best.i < 0 || score_better(o, best))) best = o;
      }
      if (lane == 0) {
        const int bi = best.i;
        best_g = bi;
        if (bi >= 0) {
          const int s = bi / N;
          chosen[bi] = 1;
          selected[(size_t)s * gamma_max + cnt[s]] = bi - s * N;
          cnt[s] = static_cast<int16_t>(cnt[s] + 1);
        }
      }
    }
    __syncthreads();
    if (best_g < 0) break;
    const uint32_t* tb = traj + (size_t)best_g * W;
    for (int w = threadIdx.x; w < W; w += blockDim.x) B[w] |= tb[w];
    __syncthreads();
  }

  // Unused slots, per-sequence unions of their own selections.
  for (int i = threadIdx.x; i < nseq * gamma_max; i += blockDim.x) {
    const int s = i / gamma_max, j = i - s * gamma_max;
    if (j >= cnt[s]) selected[i] = -1;
  }
  for (int s = warp; s < nseq; s += nwarps) {
    int c = 0;
    for (int w = lane; w < W; w += 32) {
      uint32_t u = 0;
      for (int j = 0; j < cnt[s]; ++j) u |= traj[(size_t)(s * N + selected[(size_t)s * gamma_max + j]) * W + w];
      c += __popc(u);
    }
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    if (lane == 0) union_size[s] = c;
  }
  if (pred_B)  // the batch's one buffer in row 0, the other rows empty
    for (int i = threadIdx.x; i < nseq * W; i += blockDim.x) pred_B[i] = i < W ? B[i] : 0u;
  if (verify_rows && threadIdx.x == 0) {
    int tok = 0;
    for (int s = 0; s < nseq; ++s) {
      for (int q = 0; q <= cnt[s]; ++q, ++tok) {
        if (tok >= T_expected) continue;
        const int node = q == 0 ? -1 : selected[(size_t)s * gamma_max + q - 1];
        verify_rows[tok] = s * (N + 1) + (q == 0 ? 0 : 1 + node);
        verify_conf[tok] = q == 0 ? 1.f : P[(size_t)s * N + node];
      }
    }
    if (tok != T_expected) flag_error(dev_err, MOE_DEV_CAPACITY);
  }
}

}  // namespace

// s with eps == 2^-s (0 <= s <= 20), or -1.
int eps_shift(float eps) {
  for (int q = 0; q <= 20; ++q)
    if (eps == static_cast<float>(1.0 / static_cast<double>(1u << q))) return q;
  return -1;
}

int eco_validate(const eco_cfg& c, int nseq) {
  if (nseq < 0 || c.N < 1 || c.N > kMaxN || c.W < 1 || c.W > kMaxW) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(c.N) * c.W > kMaxNW) return MOE_ERR_UNSUPPORTED;
  if (c.gamma_max < 0 || c.mode < 0 || c.mode > 2) return MOE_ERR_ARG;
  if (c.mode == 2 && (static_cast<long long>(nseq) * c.N > kMaxN ||
                      static_cast<long long>(nseq) * c.N * c.W > kMaxNW))
    return MOE_ERR_UNSUPPORTED;
  // eps must be 2^-s, 0 <= s <= 20, and W*32 * 2^s < 2^29 so that
  // X = c * 2^s + 1 fits in 29 bits and P's significand times X in 53.
  const int s = eps_shift(c.eps);
  if (s < 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<double>(c.W) * 32.0 * static_cast<double>(1u << s) >= 536870912.0)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int eco_launch(const EcoArgs& a) {
  if (a.nseq == 0) return MOE_OK;
  const auto& c = a.cfg;
  if (c.mode == 2) {
    const size_t smem = (static_cast<size_t>(a.nseq) * c.N * c.W + c.W) * sizeof(uint32_t);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(eco_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    LaunchScope ls(kProfEco, a.stream);
    eco_batch_kernel<<<1, 512, smem, a.stream>>>(a.P, a.parent, a.own_fp, a.gamma, c.N, c.W, a.nseq, c.gamma_max,
                                                  eps_shift(c.eps), a.selected, a.union_size, a.dev_err,
                                                  a.verify_rows, a.verify_conf, a.T_expected, a.ready_flag,
                                                  a.pred_B);
    return check_launch();
  }
  size_t smem = (static_cast<size_t>(c.N) * c.W + c.W) * sizeof(uint32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(eco_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int threads = c.W >= 256 || c.N >= 16 ? 512 : 256;
  LaunchScope ls(kProfEco, a.stream);
  eco_kernel<<<a.nseq, threads, smem, a.stream>>>(a.P, a.parent, a.own_fp, a.gamma, c.N, c.W,
                                                  c.gamma_max, c.mode, eps_shift(c.eps),
                                                  (static_cast<long long>(c.W) * 32) << eps_shift(c.eps) < (1ll << 24) - 1,
                                                  a.selected, a.union_size, a.dev_err,
                                                  a.verify_rows, a.verify_conf, a.T_expected,
                                                  a.nseq, a.ready_flag, a.pred_B);
  return check_launch();
}

}  // namespace moe

extern "C" int eco_select(const float* P, const int32_t* parent, const uint32_t* own_fp,
                          int32_t nseq, const int32_t* gamma_per_seq, const eco_cfg* cfg,
                          int32_t* selected, int32_t* union_size, int32_t* dev_err, void* stream) {
  if (!cfg) return MOE_ERR_ARG;
  int st = moe::eco_validate(*cfg, nseq);
  if (st != MOE_OK) return st;
  if (nseq > 0 && (!P || !parent || !own_fp || !union_size || (cfg->gamma_max > 0 && !selected)))
    return MOE_ERR_ARG;
  moe::EcoArgs a{P, parent, own_fp, nseq, gamma_per_seq, *cfg, selected, union_size, dev_err,
                 nullptr, nullptr, 0, static_cast<cudaStream_t>(stream), nullptr, nullptr};
  return moe::eco_launch(a);
}
