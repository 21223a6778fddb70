// L2 prefetch of the next layer's predicted experts (see NextLayerPrefetch),
// shared by the tensor-core down kernels.
#pragma once

#include "common.cuh"

namespace moe {

constexpr long long kPfPiece = 32 << 10;

// Issued by one thread of CTA c of G: the predicted experts in ascending
// order, the budget split evenly over them in kPfPiece pieces from the start
// of each expert's weights, pieces dealt round-robin over the CTAs.
// Prefetching changes no result.
static __device__ __noinline__ void l2_prefetch_next_layer(const NextLayerPrefetch& pf, int E, int c, int G) {
  const int EW = (E + 31) >> 5;
  uint32_t mask[32];
  int n = 0;
  for (int w = 0; w < EW; ++w) {
    uint32_t m = 0;
    const long long b = pf.bit0 + 32ll * w;
    const long long w0 = b >> 5;
    const int sh = static_cast<int>(b & 31);
    for (int r = 0; r < pf.rows; ++r) {
      const uint32_t* row = pf.pred_B + (size_t)r * pf.W;
      const uint32_t lo = w0 < pf.W ? row[w0] : 0u;
      const uint32_t hi = (sh && w0 + 1 < pf.W) ? row[w0 + 1] : 0u;
      m |= sh ? (lo >> sh) | (hi << (32 - sh)) : lo;
    }
    const int valid = E - 32 * w;
    if (valid < 32) m &= (1u << valid) - 1u;
    mask[w] = m;
    n += __popc(m);
  }
  if (n == 0) return;
  long long ppe = pf.budget / n / kPfPiece;  // pieces per expert
  const long long cap = (pf.expert_bytes + kPfPiece - 1) / kPfPiece;
  if (ppe > cap) ppe = cap;
  for (long long i = c; i < n * ppe; i += G) {
    int j = static_cast<int>(i / ppe);
    const long long off = (i % ppe) * kPfPiece;
    int e = -1;
    for (int w = 0; w < EW && e < 0; ++w) {
      const int cnt = __popc(mask[w]);
      if (j < cnt) {
        uint32_t mm = mask[w];
        for (int q = 0; q < j; ++q) mm &= mm - 1;
        e = 32 * w + __ffs(mm) - 1;
      } else {
        j -= cnt;
      }
    }
    if (e < 0 || off >= pf.expert_bytes) continue;
    const long long sz = pf.expert_bytes - off < kPfPiece ? pf.expert_bytes - off : kPfPiece;
    const uint8_t* a = pf.base + e * pf.expert_bytes + off;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(static_cast<uint32_t>(sz)) : "memory");
  }
}

}  // namespace moe
