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

// Shared memory is sized to T and E (a few KB in verify steps), so the head
// can sit next to a running FFN CTA and start as soon as it is launched.
template <int NPL>
__global__ void __launch_bounds__(256) layer_head_kernel(RouteArgs ra, int32_t* n_unique, int32_t* unique,
                                                         int32_t* offsets, int32_t* perm_token, int32_t* perm_slot,
                                                         int32_t* inv, float* reuse_ratio) {
  extern __shared__ __align__(16) uint8_t head_smem[];
  const moe_route_cfg& c = ra.cfg;
  const int TK = c.T * c.k;
  const size_t bias_bytes = (routing::bias_view_bytes(c.T, c.E) + 15) & ~size_t(15);
  const size_t union_bytes = (unions::union_view_bytes(c.E) + 15) & ~size_t(15);
  routing::BiasView bv = routing::carve_bias(head_smem, c.T, c.E);
  unions::UnionView uv = unions::carve_union(head_smem + bias_bytes, c.E);
  // The routing result stays in shared memory for the union; a copy goes out.
  int32_t* s_ids = reinterpret_cast<int32_t*>(head_smem + bias_bytes + union_bytes);
  float* s_w = reinterpret_cast<float*>(s_ids + TK);

  // The logits rows are inputs, not results of the previous kernel: pull
  // them towards L2 while that kernel finishes.  (The row map may still be
  // in flight for the first layer, so every index is bounds-checked first;
  // a prefetch only moves data, it never changes results.)
  {
    const int lines = (c.E * 4 + 127) / 128;
    for (int i = threadIdx.x; i < c.T * lines; i += blockDim.x) {
      const int t = i / lines;
      const long long row = ra.rows ? ra.rows[t] : t;
      if (row >= 0 && (!ra.rows || row < ra.rows_limit))
        asm volatile("prefetch.global.L2 [%0];" ::"l"(ra.logits + row * c.E + (i - t * lines) * 32));
    }
  }
  pdl_wait();
  pdl_trigger();
  if (c.use_bias)
    routing::route_bias_block<NPL>(ra.logits, ra.rows, ra.rows_limit, ra.w_conf, c.T, c.E, c.k, c.cap, c.alpha,
                                   s_ids, s_w, ra.dev_err, bv);
  else
    routing::route_plain_warps<NPL>(ra.logits, ra.rows, ra.rows_limit, c.T, c.E, c.k, s_ids, s_w, ra.dev_err,
                                    threadIdx.x >> 5, blockDim.x >> 5);
  __syncthreads();
  for (int i = threadIdx.x; i < TK; i += blockDim.x) {
    ra.ids[i] = s_ids[i];
    ra.w[i] = s_w[i];
  }
  unions::union_block(s_ids, c.T, c.k, c.E, bv.member, uv, n_unique, unique, offsets, perm_token, perm_slot, inv,
                      reuse_ratio, ra.dev_err);
}

template <int NPL>
int launch_npl(const RouteArgs& ra, int32_t* n_unique, int32_t* unique, int32_t* offsets, int32_t* perm_token,
               int32_t* perm_slot, int32_t* inv, float* reuse_ratio, bool pdl) {
  const size_t smem = ((routing::bias_view_bytes(ra.cfg.T, ra.cfg.E) + 15) & ~size_t(15)) +
                      ((unions::union_view_bytes(ra.cfg.E) + 15) & ~size_t(15)) +
                      static_cast<size_t>(ra.cfg.T) * ra.cfg.k * 8;
  if (smem > 48 * 1024 && cudaFuncSetAttribute(layer_head_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  LaunchScope ls(kProfRoute, ra.stream);
  return launch_k(layer_head_kernel<NPL>, dim3(1), dim3(256), smem, ra.stream, pdl, ra, n_unique, unique, offsets,
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
