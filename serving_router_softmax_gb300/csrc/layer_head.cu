// Fused per-layer head of the verify step: routing (optionally with the
// S2-MoE reuse bias) followed by the expert union and token permutation, in
// one single-CTA launch.  Same arithmetic and outputs as moe_route followed by
// moe_union_permute (EcoSpec write-up section 3.1 and section 2; S2-MoE
// write-up component 2, steps 1-3, and challenge 2), laid out for latency:
//   - shared state is cleared, and (once the row map is complete) each warp's
//     logits row is loaded, before the wait on the previous kernel: the
//     logits are step inputs, not results of that kernel;
//   - the routing rounds record the union bookkeeping (token x expert bits,
//     group sizes) as they select, so the union needs no scatter pass;
//   - with the bias, g_e is one expert per thread and E* a rank test (an
//     expert is in E* when fewer than cap experts beat it), with no serial
//     selection rounds;
//   - optionally (bf16 tensor-core layers with T <= 32), extra CTAs copy the
//     token rows for the FFN and zero its fix-up counters, and CTA 0
//     publishes the union to the gate/up kernel (release store) as soon as
//     it is written, so that kernel can start its weight stream while this
//     one finishes the permutation.
// Launched with programmatic dependent launch, so its launch overlaps the
// previous layer's last kernel.
#include "common.cuh"
#include "route_dev.cuh"
#include "fp8_quant.cuh"

namespace moe {
namespace {

using routing::kFull;
using routing::Row;

constexpr int kHeadThreads = 256;
constexpr int kHeadWarps = kHeadThreads / 32;

struct HeadSmem {
  int32_t* count;     // [EP] group sizes, EP = 32 * ceil(E / 32) (16-byte aligned, zero past E)
  int32_t* ustart;    // [E] first perm position of each expert's group
  uint32_t* cand_key; // [E] experts with g_e > 0: order keys ... (bias only)
  int32_t* cand_e;    // [E] ... and ids, in arbitrary order
  uint32_t* member;   // [T][EW] routed experts per token (union bookkeeping)
  uint32_t* member0;  // [T][EW] unbiased top-k per token (bias only)
  int32_t* ids;       // [T*k]
  float* w;           // [T*k]
  float* v1;          // [T] top-1 logit (bias only)
  float* vk1;         // [T] (k+1)-th logit (bias only)
  float* wc;          // [T] confidence weights (bias only)
  float* vw;          // [T] the weight a token adds to g_e: wc, or 0 if its row is unusable
  uint32_t* estar;    // [EW] preferred experts (bias only)
  uint8_t* bad;       // [T] 0 ok, 1 NaN logit, 2 row outside the node table
  int* err;
  int* ncand;
};

__host__ __device__ inline size_t head_smem_bytes(int T, int E, int k) {
  const int EW = (E + 31) / 32;
  const size_t EP = 32 * static_cast<size_t>(EW);
  return 4 * (EP + 3 * static_cast<size_t>(E) + 2 * static_cast<size_t>(T) * EW + 2 * static_cast<size_t>(T) * k +
              4 * static_cast<size_t>(T) + EW + 2) +
         ((static_cast<size_t>(T) + 15) & ~size_t(15));
}

__device__ __forceinline__ HeadSmem carve(uint8_t* p, int T, int E, int k) {
  const int EW = (E + 31) / 32;
  HeadSmem s;
  s.count = reinterpret_cast<int32_t*>(p);
  s.ustart = s.count + 32 * EW;
  s.cand_key = reinterpret_cast<uint32_t*>(s.ustart + E);
  s.cand_e = reinterpret_cast<int32_t*>(s.cand_key + E);
  s.member = reinterpret_cast<uint32_t*>(s.cand_e + E);
  s.member0 = s.member + (size_t)T * EW;
  s.ids = reinterpret_cast<int32_t*>(s.member0 + (size_t)T * EW);
  s.w = reinterpret_cast<float*>(s.ids + (size_t)T * k);
  s.v1 = s.w + (size_t)T * k;
  s.vk1 = s.v1 + T;
  s.wc = s.vk1 + T;
  s.vw = s.wc + T;
  s.estar = reinterpret_cast<uint32_t*>(s.vw + T);
  s.err = reinterpret_cast<int*>(s.estar + EW);
  s.ncand = s.err + 1;
  s.bad = reinterpret_cast<uint8_t*>(s.ncand + 1);
  return s;
}

// Top-k of a loaded row, softmax over the selected logits, and the union
// bookkeeping of the selected experts.  Lane j keeps slot j.
template <int NPL>
__device__ __forceinline__ void select_token(Row<NPL>& r, int t, int E, int k, int EW, int lane, HeadSmem& sm) {
  float mine_v = -INFINITY, m = 0.f;
  int mine_i = -1;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv;
    int bi;
    routing::argmax_round(r, E, lane, bv, bi);
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
    sm.ids[t * k + lane] = mine_i;
    sm.w[t * k + lane] = __fdiv_rn(ex, s);
    // a token's k ids are distinct (each round excludes the earlier picks);
    // k <= E is checked on the host, so every round finds an expert
    if (mine_i >= 0 && mine_i < E) {
      atomicOr(&sm.member[t * EW + (mine_i >> 5)], 1u << (mine_i & 31));
      atomicAdd(&sm.count[mine_i], 1);
    }
  }
}

__device__ __forceinline__ void invalid_token(int t, int k, int lane, int bad, HeadSmem& sm, int32_t* dev_err) {
  if (lane == 0) flag_error(dev_err, bad == 2 ? MOE_DEV_CAPACITY : MOE_DEV_NAN_LOGIT);
  for (int j = lane; j < k; j += 32) {
    sm.ids[t * k + j] = -1;
    sm.w[t * k + j] = 0.f;
  }
  if (lane == 0) *sm.err = MOE_DEV_BAD_ID;  // the union is undefined without every token's ids
}

template <int NPL>
__global__ void __launch_bounds__(kHeadThreads) layer_head_kernel(RouteArgs ra, int32_t* n_unique, int32_t* unique,
                                                                  int32_t* offsets, int32_t* perm_token,
                                                                  int32_t* perm_slot, int32_t* inv,
                                                                  float* reuse_ratio, int rows_ready,
                                                                  HeadPrep hp) {
  extern __shared__ __align__(16) uint8_t head_smem[];
  if (blockIdx.x > 0) {
    // ---- FFN prep CTAs.  When this grid starts, the previous layer's FFN
    // kernels have finished (the kernel it follows starts it only after its
    // own wait), so the token rows and counters are free to overwrite; only
    // the row map may still be in flight (first layer).
    if (!rows_ready) pdl_wait();
    const long long nth = (long long)(gridDim.x - 1) * blockDim.x;
    const long long tid = (long long)(blockIdx.x - 1) * blockDim.x + threadIdx.x;
    for (long long i = tid; i < hp.n_counters; i += nth) hp.counters[i] = 0;
    if (hp.xq_hi) {
      // FP8 layers: one CTA per token row quantizes it (max |x|, power-of-two
      // scale, hi/lo E4M3 rows); padding rows up to q_rows get scale 1.
      __shared__ float s_max[kHeadThreads / 32];
      for (int t = blockIdx.x - 1; t < hp.q_rows; t += gridDim.x - 1) {
        const long long row = t < ra.cfg.T ? hp.x_rows[t] : -1;
        const bool ok = t < ra.cfg.T && row >= 0 && row < hp.x_rows_limit;
        if (t < ra.cfg.T && !ok && threadIdx.x == 0) flag_error(ra.dev_err, MOE_DEV_BAD_ID);
        fp8q::quantize_row(ok ? hp.x + (size_t)row * hp.H : nullptr, hp.H, hp.xq_hi + (size_t)t * hp.H,
                           hp.xq_lo + (size_t)t * hp.H, t < ra.cfg.T ? hp.xscale + t : nullptr, s_max,
                           t < ra.cfg.T);
        if (t >= ra.cfg.T && threadIdx.x == 0) hp.xscale[t] = 1.f;
      }
      return;
    }
    const int cpr = hp.H / 8;  // 16-byte chunks per row
    for (long long i = tid; i < (long long)ra.cfg.T * cpr; i += nth) {
      const int t = static_cast<int>(i / cpr);
      const int ch = static_cast<int>(i - (long long)t * cpr);
      const long long row = hp.x_rows[t];
      if (row >= 0 && row < hp.x_rows_limit)
        *reinterpret_cast<uint4*>(hp.xd + (size_t)t * hp.H + ch * 8) =
            *reinterpret_cast<const uint4*>(hp.x + (size_t)row * hp.H + ch * 8);
      else
        flag_error(ra.dev_err, MOE_DEV_BAD_ID);
    }
    return;
  }
  const moe_route_cfg& c = ra.cfg;
  const int T = c.T, E = c.E, k = c.k, TK = T * k;
  const int EW = (E + 31) >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  HeadSmem sm = carve(head_smem, T, E, k);

  // ---- before the dependency wait: clear the bookkeeping, fetch the rows.
  for (int i = threadIdx.x; i < 2 * T * EW; i += kHeadThreads) sm.member[i] = 0;  // member and member0
  for (int e = threadIdx.x; e < 32 * EW; e += kHeadThreads) sm.count[e] = 0;
  for (int i = threadIdx.x; i < EW; i += kHeadThreads) sm.estar[i] = 0;
  if (threadIdx.x == 0) {
    *sm.err = 0;
    *sm.ncand = 0;
  }
  // One token per warp keeps its row in registers through both passes.
  const bool keep = T <= kHeadWarps;
  Row<NPL> kept;
  kept.taken = 0;
  bool kept_nan = false, loaded = false;
  int kept_bad = 0;
  auto row_of = [&](int t, int& bad) -> long long {
    const long long row = ra.rows ? ra.rows[t] : t;
    bad = (ra.rows && (row < 0 || row >= ra.rows_limit)) ? 2 : 0;
    return row;
  };
  int my_bad = 0;
  auto load_conf = [&]() {
    for (int t = threadIdx.x; t < T; t += kHeadThreads) {
      const float cf = ra.w_conf[t];
      sm.wc[t] = cf;
      if (!(cf >= 0.f)) my_bad = 1;  // NaN or negative
    }
  };
  if (rows_ready && c.use_bias) load_conf();
  if (keep && rows_ready) {
    if (warp < T) {
      const long long row = row_of(warp, kept_bad);
      if (!kept_bad) kept_nan = routing::load_row<NPL>(ra.logits + row * E, E, lane, kept, nullptr, 0.f);
      loaded = true;
    }
  } else {
    // Warm L2 with bounds-checked addresses only: the row map may still be
    // in flight (it is written by the kernel before the first layer's head),
    // and a prefetch never changes results.
    const int lines = (E * 4 + 127) / 128;
    for (int i = threadIdx.x; i < T * lines; i += kHeadThreads) {
      const int t = i / lines;
      const long long row = ra.rows ? ra.rows[t] : t;
      if (row >= 0 && (!ra.rows || row < ra.rows_limit))
        asm volatile("prefetch.global.L2 [%0];" ::"l"(ra.logits + row * E + (i - t * lines) * 32));
    }
  }
  pdl_wait();
  pdl_trigger();
  if (keep && !loaded && warp < T) {
    const long long row = row_of(warp, kept_bad);
    if (!kept_bad) kept_nan = routing::load_row<NPL>(ra.logits + row * E, E, lane, kept, nullptr, 0.f);
  }
  if (c.use_bias && !rows_ready) load_conf();
  __syncthreads();  // bookkeeping cleared

  if (c.use_bias) {
    // ---- pass 1: unbiased top-(k+1) -> TopK membership, l_(1), l_(k+1)
    for (int t = warp; t < T; t += kHeadWarps) {
      Row<NPL> r;
      int bad = 0;
      bool nan = false;
      if (keep) {
        r = kept;
        bad = kept_bad;
        nan = kept_nan;
      } else {
        const long long row = row_of(t, bad);
        if (!bad) nan = routing::load_row<NPL>(ra.logits + row * E, E, lane, r, nullptr, 0.f);
      }
      if (!bad && nan) bad = 1;
      if (lane == 0) {
        sm.bad[t] = static_cast<uint8_t>(bad);
        sm.vw[t] = bad ? 0.f : sm.wc[t];
      }
      if (bad) continue;
      // The round results stay in registers (lane j keeps the j-th id) and
      // reach shared memory after the rounds, so that no lane branches off
      // between the warp reductions.
      float v1 = 0.f, vk1 = 0.f;
      int mine = -1;
      __syncwarp();
#pragma unroll 1
      for (int j = 0; j <= k; ++j) {
        float bv;
        int bi;
        routing::argmax_round(r, E, lane, bv, bi);
        v1 = j == 0 ? bv : v1;
        vk1 = bv;
        mine = (lane == j && j < k) ? bi : mine;
      }
      if (lane == 0) {
        sm.v1[t] = v1;
        sm.vk1[t] = vk1;
      }
      if (mine >= 0 && mine < E) atomicOr(&sm.member0[t * EW + (mine >> 5)], 1u << (mine & 31));
    }
    const bool conf_bad = __syncthreads_or(my_bad) != 0;
    if (conf_bad) {
      if (threadIdx.x == 0) flag_error(ra.dev_err, MOE_DEV_BAD_PROB);
      for (int i = threadIdx.x; i < TK; i += kHeadThreads) {
        ra.ids[i] = -1;
        ra.w[i] = 0.f;
      }
      if (threadIdx.x == 0) {
        flag_error(ra.dev_err, MOE_DEV_BAD_ID);
        *n_unique = 0;
        *reuse_ratio = 0.f;
        offsets[0] = 0;
        if (hp.ready_flag) st_release_gpu(hp.ready_flag, hp.ready_value);  // union size 0
      }
      return;
    }
    // ---- g_e (fp32, tokens in ascending order, plain adds), one expert per
    // thread.  A token that does not hold e, or whose row was unusable (vw =
    // 0), adds +0.0, which leaves every partial sum unchanged (sums are never
    // -0.0).  Experts with g_e > 0 (at most T*k of them) become candidates.
    for (int e = threadIdx.x; e < E; e += kHeadThreads) {
      const int we = e >> 5;
      const uint32_t bit = 1u << (e & 31);
      float acc = 0.f;
#pragma unroll 4
      for (int b = 0; b < T; ++b) acc = __fadd_rn(acc, (sm.member0[b * EW + we] & bit) ? sm.vw[b] : 0.f);
      if (acc > 0.f) {
        const int i = atomicAdd(sm.ncand, 1);
        sm.cand_key[i] = routing::order_key(acc);
        sm.cand_e[i] = e;
      }
    }
    __syncthreads();
    // ---- E* = the top-cap experts by g among g > 0 (ties to the lower id):
    // a candidate is in E* when fewer than cap candidates beat it in that
    // order (the candidates' order in the list does not matter).
    {
      const int nc = *sm.ncand;
      for (int i = threadIdx.x; i < nc; i += kHeadThreads) {
        const uint32_t ke = sm.cand_key[i];
        const int e = sm.cand_e[i];
        int b0 = 0, b1 = 0;
        int q = 0;
        for (; q + 1 < nc; q += 2) {
          const uint32_t k0 = sm.cand_key[q], k1 = sm.cand_key[q + 1];
          const int e0 = sm.cand_e[q], e1 = sm.cand_e[q + 1];
          b0 += (k0 > ke) || (k0 == ke && e0 < e);
          b1 += (k1 > ke) || (k1 == ke && e1 < e);
        }
        if (q < nc) b0 += (sm.cand_key[q] > ke) || (sm.cand_key[q] == ke && sm.cand_e[q] < e);
        if (b0 + b1 < c.cap) atomicOr(&sm.estar[e >> 5], 1u << (e & 31));
      }
    }
    __syncthreads();
    // ---- pass 2: route the biased logits l' = l + lam_b on E*
    for (int t = warp; t < T; t += kHeadWarps) {
      if (sm.bad[t]) {
        invalid_token(t, k, lane, sm.bad[t], sm, ra.dev_err);
        continue;
      }
      const float lam = __fmul_rn(c.alpha, __fsub_rn(sm.v1[t], sm.vk1[t]));
      Row<NPL> r;
      if (keep) {
        // from the kept keys: key_value(order_key(x)) == x up to the sign of
        // zero, which no comparison or exponent sees
        r = kept;
        r.taken = 0;
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
          const int e = lane + 32 * j;
          if (e < E && ((sm.estar[e >> 5] >> (e & 31)) & 1u))
            r.key[j] = routing::order_key(__fadd_rn(routing::key_value(r.key[j]), lam));
        }
      } else {
        int bad = 0;
        const long long row = row_of(t, bad);
        routing::load_row<NPL>(ra.logits + row * E, E, lane, r, sm.estar, lam);
      }
      select_token<NPL>(r, t, E, k, EW, lane, sm);
    }
  } else {
    // ---- plain routing
    for (int t = warp; t < T; t += kHeadWarps) {
      Row<NPL> r;
      int bad = 0;
      bool nan = false;
      if (keep) {
        r = kept;
        bad = kept_bad;
        nan = kept_nan;
      } else {
        const long long row = row_of(t, bad);
        if (!bad) nan = routing::load_row<NPL>(ra.logits + row * E, E, lane, r, nullptr, 0.f);
      }
      if (!bad && nan) bad = 1;
      if (bad) {
        invalid_token(t, k, lane, bad, sm, ra.dev_err);
        continue;
      }
      select_token<NPL>(r, t, E, k, EW, lane, sm);
    }
  }
  __syncthreads();

  // ---- union: warp 0 scans the group sizes; the others publish ids and weights
  const int err = *sm.err;
  for (int i = threadIdx.x; i < TK; i += kHeadThreads) {
    ra.ids[i] = sm.ids[i];
    ra.w[i] = sm.w[i];
  }
  if (err) {
    if (threadIdx.x == 0) {
      flag_error(ra.dev_err, err);
      *n_unique = 0;
      *reuse_ratio = 0.f;
      offsets[0] = 0;
      if (hp.ready_flag) st_release_gpu(hp.ready_flag, hp.ready_value);  // union size 0
    }
    return;
  }
  if (warp == 0) {
    // lane l scans experts [l * per, l * per + per); the group sizes are read
    // as 16-byte vectors when per allows (no bank conflicts)
    const int per = EW;
    const int e0 = lane * per;
    int cv[NPL];
    bool vec = false;
    if constexpr (NPL >= 4) vec = (per & 3) == 0;
    if (vec) {
      if constexpr (NPL >= 4) {
#pragma unroll
        for (int i = 0; i < NPL; i += 4) {
          int4 v = make_int4(0, 0, 0, 0);
          if (i < per) v = *reinterpret_cast<const int4*>(sm.count + e0 + i);
          cv[i] = v.x;
          cv[i + 1] = v.y;
          cv[i + 2] = v.z;
          cv[i + 3] = v.w;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < NPL; ++i) cv[i] = i < per ? sm.count[e0 + i] : 0;
    }
    int nz = 0, tok = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      nz += cv[i] > 0;
      tok += cv[i];
    }
    int nz_ex = nz, tok_ex = tok;
    warp_inclusive_sum2(nz_ex, tok_ex, lane);
    nz_ex -= nz;
    tok_ex -= tok;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = e0 + i;
      if (cv[i] > 0) {  // zero past per and past E
        sm.ustart[e] = tok_ex;
        unique[nz_ex] = e;
        offsets[nz_ex] = tok_ex;
        ++nz_ex;
        tok_ex += cv[i];
      }
    }
    if (lane == 31) {
      offsets[nz_ex] = tok_ex;  // == T*k
      *n_unique = nz_ex;
      *reuse_ratio = TK > 0 ? __fdiv_rn(static_cast<float>(nz_ex), static_cast<float>(TK)) : 0.f;
    }
    // The union (n_unique, unique, offsets) is out: publish it, with its size
    // in the high 16 bits (U <= min(E, T*k) <= 1024).  The warp barrier
    // orders every lane's stores before lane 0's release.
    __syncwarp();
    const int u_total = __shfl_sync(kFull, nz_ex, 31);
    if (lane == 0 && hp.ready_flag) st_release_gpu(hp.ready_flag, hp.ready_value | (u_total << 16));
  }
  __syncthreads();
  // ---- permutation: rank of token t in expert e's group = set bits of
  // column e over tokens t' < t
  for (int p = threadIdx.x; p < TK; p += kHeadThreads) {
    const int t = p / k;
    const int j = p - t * k;
    const int e = sm.ids[p];
    const int word = e >> 5;
    const uint32_t bit = 1u << (e & 31);
    int rank = 0;
    for (int tt = 0; tt < t; ++tt) rank += (sm.member[tt * EW + word] & bit) ? 1 : 0;
    const int pos = sm.ustart[e] + rank;
    perm_token[pos] = t;
    perm_slot[pos] = j;
    inv[p] = pos;
  }
}

template <int NPL>
int launch_npl(const RouteArgs& ra, int32_t* n_unique, int32_t* unique, int32_t* offsets, int32_t* perm_token,
               int32_t* perm_slot, int32_t* inv, float* reuse_ratio, bool pdl, bool rows_ready,
               const HeadPrep* hp) {
  const size_t smem = head_smem_bytes(ra.cfg.T, ra.cfg.E, ra.cfg.k);
  if (smem > 48 * 1024 && cudaFuncSetAttribute(layer_head_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  HeadPrep h{};
  int grid = 1;
  if (hp) {
    h = *hp;
    const long long chunks = static_cast<long long>(ra.cfg.T) * (h.H / 8);
    const long long work = chunks > h.n_counters ? chunks : h.n_counters;
    long long extra = (work + kHeadThreads - 1) / kHeadThreads;
    if (h.xq_hi && extra < h.q_rows) extra = h.q_rows;  // FP8: a CTA per token row
    if (extra > 32) extra = 32;
    grid = 1 + static_cast<int>(extra);
  }
  LaunchScope ls(kProfRoute, ra.stream);
  return launch_k(layer_head_kernel<NPL>, dim3(grid), dim3(kHeadThreads), smem, ra.stream, pdl, ra, n_unique, unique,
                  offsets, perm_token, perm_slot, inv, reuse_ratio, rows_ready ? 1 : 0, h);
}

}  // namespace

// T <= 256, E <= 1024, k <= 16 (checked by the step's validation).
int layer_head_launch(const RouteArgs& ra, int32_t* n_unique, int32_t* unique, int32_t* offsets,
                      int32_t* perm_token, int32_t* perm_slot, int32_t* inv, float* reuse_ratio, bool pdl,
                      bool rows_ready, const HeadPrep* hp) {
  if (hp && (!hp->x || !hp->x_rows || !(hp->xd || hp->xq_hi) || !hp->counters || hp->H % 16)) return MOE_ERR_ARG;
  if (hp && hp->xq_hi && (!hp->xq_lo || !hp->xscale || hp->q_rows < ra.cfg.T || hp->q_rows > 32)) return MOE_ERR_ARG;
  if (ra.cfg.T < 1 || ra.cfg.T > routing::kBiasMaxT || ra.cfg.E > 1024) return MOE_ERR_UNSUPPORTED;
  const int npl = (ra.cfg.E + 31) / 32;
  if (npl <= 1)
    return launch_npl<1>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl, rows_ready, hp);
  if (npl <= 2)
    return launch_npl<2>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl, rows_ready, hp);
  if (npl <= 4)
    return launch_npl<4>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl, rows_ready, hp);
  if (npl <= 8)
    return launch_npl<8>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl, rows_ready, hp);
  if (npl <= 16)
    return launch_npl<16>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl, rows_ready, hp);
  return launch_npl<32>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl, rows_ready, hp);
}

}  // namespace moe
