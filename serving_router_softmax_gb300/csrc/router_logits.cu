// Router (gate) logits of the verify tokens: logits[t, e] = sum_h x[t, h] * W_r[e, h].
//
// S2-MoE write-up, background (a router/gate picks each token's top-k of the
// layer's E expert FFNs); EcoSpec write-up section 2 (S_l(x_t) is a function
// of the token's hidden state).  The gate is a bias-free linear layer.
//
// The matrix W_r is small (E x H: 1 MiB for E = 128, H = 4096 bf16) and the
// token count T is a handful, so the contraction is bound by one pass over
// W_r and by launch latency, not by arithmetic (T FMAs per weight).  One CTA
// per expert row e: its 128 threads split the row into 8-element groups,
// issue all of their weight loads of a chunk at once, and multiply each group
// with up to 8 tokens' activations (read from L2, where x stays resident).
// Each thread accumulates its groups in ascending order with fp32 FMAs; the
// warps then reduce with a fixed butterfly and the CTA adds the 4 warp sums
// in warp order, so the result never depends on timing.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouterWarps = 4;
constexpr int kRouterThreads = kRouterWarps * kWarp;
constexpr int kTokPass = 8;  // tokens per pass over the row
constexpr int kChunk = 4;    // 8-element groups per thread whose loads are in flight together

__device__ __forceinline__ void load8(const uint16_t* p, float v[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8(const float* p, float v[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename XT, typename WT>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(const XT* __restrict__ x, const WT* __restrict__ w, int T, int H, int E,
              float* __restrict__ logits) {
  __shared__ float part[kRouterWarps][kTokPass];
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n8 = H >> 3;
  const WT* wrow = w + static_cast<size_t>(e) * H;
  pdl_wait();
  pdl_trigger();

  for (int t0 = 0; t0 < T; t0 += kTokPass) {
    const int nt = min(kTokPass, T - t0);
    float acc[kTokPass];
#pragma unroll
    for (int j = 0; j < kTokPass; ++j) acc[j] = 0.f;

    for (int g0 = tid; g0 < n8; g0 += kRouterThreads * kChunk) {
      float wv[kChunk][8];
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const int g = g0 + c * kRouterThreads;
        if (g < n8) {
          load8(wrow + static_cast<size_t>(g) * 8, wv[c]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) wv[c][i] = 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < kTokPass; ++j) {
        if (j < nt) {
          const XT* xr = x + static_cast<size_t>(t0 + j) * H;
#pragma unroll
          for (int c = 0; c < kChunk; ++c) {
            const int g = g0 + c * kRouterThreads;
            if (g < n8) {
              float xv[8];
              load8(xr + static_cast<size_t>(g) * 8, xv);
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[j] = fmaf(xv[i], wv[c][i], acc[j]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kTokPass; ++j) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kTokPass; ++j) part[warp][j] = acc[j];
    }
    __syncthreads();
    if (tid < nt) {
      float s = part[0][tid];
#pragma unroll
      for (int q = 1; q < kRouterWarps; ++q) s += part[q][tid];
      logits[static_cast<size_t>(t0 + tid) * E + e] = s;
    }
    __syncthreads();
  }
}

template <typename XT, typename WT>
int router_go(const RouterArgs& a) {
  LaunchScope ls(kProfRouter, a.stream);
  return launch_k(router_kernel<XT, WT>, dim3(a.cfg.E), dim3(kRouterThreads), 0, a.stream, a.pdl,
                  static_cast<const XT*>(a.x), static_cast<const WT*>(a.w_router), a.cfg.T, a.cfg.H,
                  a.cfg.E, a.logits);
}

}  // namespace

int router_validate(const moe_router_cfg& c) {
  if (c.T < 0 || c.H <= 0 || c.E <= 0) return MOE_ERR_ARG;
  if (c.H % 8 != 0 || c.H > (1 << 20) || c.E > 1024 || c.T > 65536) return MOE_ERR_UNSUPPORTED;
  const bool xd = c.x_dtype == MOE_DTYPE_F32 || c.x_dtype == MOE_DTYPE_BF16;
  const bool wd = c.w_dtype == MOE_DTYPE_F32 || c.w_dtype == MOE_DTYPE_BF16;
  return xd && wd ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

int router_launch(const RouterArgs& a) {
  const bool xb = a.cfg.x_dtype == MOE_DTYPE_BF16, wb = a.cfg.w_dtype == MOE_DTYPE_BF16;
  if (xb && wb) return router_go<uint16_t, uint16_t>(a);
  if (xb) return router_go<uint16_t, float>(a);
  if (wb) return router_go<float, uint16_t>(a);
  return router_go<float, float>(a);
}

}  // namespace moe

extern "C" int moe_router_logits(const void* x, const void* w_router, const moe_router_cfg* cfg,
                                 float* logits, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_ARG;
  const int st = router_validate(*cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !w_router || !logits) return MOE_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(w_router) % 16 ||
      reinterpret_cast<uintptr_t>(logits) % 4)
    return MOE_ERR_ARG;
  RouterArgs a{x, w_router, *cfg, logits, static_cast<cudaStream_t>(stream), false};
  const int r = router_launch(a);
  return r != MOE_OK ? r : check_launch();
}
