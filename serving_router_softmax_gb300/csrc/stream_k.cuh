// Stream-K bookkeeping shared by the tensor-core FFN kernels.
//
// A launch splits the layer's pipeline units (KU per 128-row tile) evenly:
// CTA c owns units [s0, s1).  A tile cut between CTAs is finished by the
// last of them to arrive, which sums every contributor's fp32 partials in
// CTA order, so results do not depend on timing or on the order in which a
// CTA walks its own tiles.
#pragma once

namespace moe {

// The CTA that owns unit x when `total` units are split over G CTAs.
__device__ __forceinline__ long long seg_owner(long long x, long long total, int G) {
  return ((x + 1) * G - 1) / total;
}

// The tiles a CTA touches, one segment each, in the order it processes
// them.  With split_first, the split ones come first (its first and last
// tile, when it owns only part of them), then the whole tiles in ascending
// order: the fix-up of a shared tile then happens while the CTA still
// streams weights, and the CTA ends on a whole tile, whose epilogue needs no
// partials, no atomic and no reads of other CTAs' sums (measured faster for
// the bf16 kernels).  Without it, plain ascending order (measured faster
// for the FP8 kernels, whose per-k-block epilogue is busier early on).
// Every role of the CTA walks the same order.
struct Segments {
  long long s0, s1;
  int KU, t_first, n_first, n_last, n;

  __device__ __forceinline__ void init(long long a, long long b, int ku, bool split_first) {
    s0 = a;
    s1 = b;
    KU = ku;
    n = n_first = n_last = t_first = 0;
    if (b <= a || ku <= 0) return;
    t_first = static_cast<int>(a / ku);
    const int t_last = static_cast<int>((b - 1) / ku);
    n = t_last - t_first + 1;
    if (!split_first) return;
    n_first = (a > static_cast<long long>(t_first) * ku || b < static_cast<long long>(t_first + 1) * ku) ? 1 : 0;
    n_last = (n > 1 && b < static_cast<long long>(t_last + 1) * ku) ? 1 : 0;
  }
  // Segment i in processing order: tile t, units [u0, u1) of it.
  __device__ __forceinline__ void get(int i, int& t, int& u0, int& u1) const {
    if (i < n_first)
      t = t_first;
    else if (i < n_first + n_last)
      t = t_first + n - 1;
    else
      t = t_first + n_first + (i - n_first - n_last);
    const long long base = static_cast<long long>(t) * KU;
    u0 = static_cast<int>(s0 > base ? s0 - base : 0);
    u1 = static_cast<int>(s1 < base + KU ? s1 - base : KU);
  }
};

}  // namespace moe
