// moe_route: router top-k + softmax weights, with the optional S2-MoE
// reuse-aware soft bias (kernels; the arithmetic is in route_dev.cuh).
//
// Routing follows the EcoSpec write-up, section 3.1; the bias follows the
// S2-MoE write-up, component 2 (confidence-weighted expert importance g_e, a
// bounded preferred set E* of the top `cap` experts, and an additive per-token
// bias proportional to the margin between the top-1 and (k+1)-th logits).
// The biased variant runs in a single CTA because g_e aggregates all tokens.
#include "common.cuh"
#include "route_dev.cuh"

namespace moe {
namespace {

using namespace routing;

template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits,
                                                    const int32_t* __restrict__ rows, int rows_limit,
                                                    int T, int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w, int32_t* dev_err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  route_plain_warps<NPL>(logits, rows, rows_limit, T, E, k, ids, w, dev_err, warp, nwarps);
}

// Single-CTA biased routing; 8 warps loop over the tokens.
template <int NPL>
__global__ void __launch_bounds__(256) route_bias_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ rows, int rows_limit,
    const float* __restrict__ w_conf, int T, int E, int k, int cap, float alpha,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* dev_err) {
  __shared__ BiasSmem sm;
  route_bias_block<NPL>(logits, rows, rows_limit, w_conf, T, E, k, cap, alpha, ids, w, dev_err, view_of(sm));
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
