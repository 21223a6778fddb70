// Fused per-layer head of the verify step: routing (optionally with the
// S2-MoE reuse bias) followed by the expert union and token permutation, in
// one single-CTA launch.  Same arithmetic as moe_route + moe_union_permute
// (route_dev.cuh, union_dev.cuh); launched with programmatic dependent launch
// so that its launch overlaps the previous layer's last kernel.
#include "common.cuh"
#include "route_dev.cuh"
#include "union_dev.cuh"

namespace moe {
namespace {

template <int NPL>
__global__ void __launch_bounds__(256) layer_head_kernel(RouteArgs ra, int32_t* n_unique, int32_t* unique,
                                                         int32_t* offsets, int32_t* perm_token, int32_t* perm_slot,
                                                         int32_t* inv, float* reuse_ratio) {
  __shared__ routing::BiasSmem bs;  // its membership bitmap is reused by the union
  __shared__ unions::UnionSmem us;
  pdl_wait();
  pdl_trigger();
  const moe_route_cfg& c = ra.cfg;
  if (c.use_bias)
    routing::route_bias_block<NPL>(ra.logits, ra.rows, ra.rows_limit, ra.w_conf, c.T, c.E, c.k, c.cap, c.alpha,
                                   ra.ids, ra.w, ra.dev_err, bs);
  else
    routing::route_plain_warps<NPL>(ra.logits, ra.rows, ra.rows_limit, c.T, c.E, c.k, ra.ids, ra.w, ra.dev_err,
                                    threadIdx.x >> 5, blockDim.x >> 5);
  __syncthreads();
  unions::union_block(ra.ids, c.T, c.k, c.E, bs.member, us, n_unique, unique, offsets, perm_token, perm_slot, inv,
                      reuse_ratio, ra.dev_err);
}

template <int NPL>
int launch_npl(const RouteArgs& ra, int32_t* n_unique, int32_t* unique, int32_t* offsets, int32_t* perm_token,
               int32_t* perm_slot, int32_t* inv, float* reuse_ratio, bool pdl) {
  LaunchScope ls(kProfRoute, ra.stream);
  return launch_k(layer_head_kernel<NPL>, dim3(1), dim3(256), 0, ra.stream, pdl, ra, n_unique, unique, offsets,
                  perm_token, perm_slot, inv, reuse_ratio);
}

}  // namespace

// T <= 256, E <= 1024 (checked by the step's validation).
int layer_head_launch(const RouteArgs& ra, int32_t* n_unique, int32_t* unique, int32_t* offsets,
                      int32_t* perm_token, int32_t* perm_slot, int32_t* inv, float* reuse_ratio, bool pdl) {
  if (ra.cfg.T < 1 || ra.cfg.T > routing::kBiasMaxT || ra.cfg.E > 1024) return MOE_ERR_UNSUPPORTED;
  const int npl = (ra.cfg.E + 31) / 32;
  if (npl <= 1) return launch_npl<1>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl);
  if (npl <= 2) return launch_npl<2>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl);
  if (npl <= 4) return launch_npl<4>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl);
  if (npl <= 8) return launch_npl<8>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl);
  if (npl <= 16) return launch_npl<16>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl);
  return launch_npl<32>(ra, n_unique, unique, offsets, perm_token, perm_slot, inv, reuse_ratio, pdl);
}

}  // namespace moe
