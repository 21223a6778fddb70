// E4M3 helpers shared by the FP8 expert FFN and the layer head that
// quantizes its token rows.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace moe {
namespace fp8q {

constexpr float kLoScale = 16.f;

__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}

__device__ __forceinline__ uint8_t float_to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Splits v (already divided by its scale, |v| <= 448) into hi + lo / 16.
__device__ __forceinline__ void split_e4m3(float v, uint8_t& hi, uint8_t& lo) {
  hi = float_to_e4m3(v);
  lo = float_to_e4m3((v - e4m3_to_float(hi)) * kLoScale);
}

// Power-of-two scale s with amax / s in [128, 256), and 1/s: dividing by s is
// then an exact multiplication.  Zero, NaN or tiny amax give s = 1.
__device__ __forceinline__ void pow2_scale(float amax, float& s, float& inv_s) {
  const int f = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
  if (!(amax > 0.f) || f < -119 || f > 127) {
    s = 1.f;
    inv_s = 1.f;
    return;
  }
  s = __uint_as_float(static_cast<uint32_t>(f - 7 + 127) << 23);
  inv_s = __uint_as_float(static_cast<uint32_t>(7 - f + 127) << 23);
}


// Quantizes one bf16 row of H values (x may be NULL: a zero row) into hi/lo
// E4M3 rows with the power-of-two scale of its max |x| (written to *scale
// when scale is not NULL).  Called by every thread of the block (it
// synchronises the block); s_max is blockDim.x / 32 floats of shared memory.
__device__ __forceinline__ void quantize_row(const uint16_t* __restrict__ x, int H, uint8_t* __restrict__ hi_row,
                                             uint8_t* __restrict__ lo_row, float* scale, float* s_max,
                                             bool write) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  float amax = 0.f;
  if (x)
    for (int c = tid * 8; c < H; c += blockDim.x * 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(x + c);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(wv[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(wv[i] & 0xFFFF0000u)));
      }
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  if (lane == 0) s_max[warp] = amax;
  __syncthreads();
  amax = s_max[0];
  for (int w = 1; w < nw; ++w) amax = fmaxf(amax, s_max[w]);
  float sc, inv_sc;
  pow2_scale(amax, sc, inv_sc);
  if (write) {
    for (int c = tid * 16; c < H; c += blockDim.x * 16) {
      uint32_t hw[4] = {0, 0, 0, 0}, lw[4] = {0, 0, 0, 0};
      if (x) {
        const uint4 va = *reinterpret_cast<const uint4*>(x + c);
        const uint4 vb = *reinterpret_cast<const uint4*>(x + c + 8);
        const uint32_t wv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint8_t ha, la, hb, lb;
          split_e4m3(__uint_as_float(wv[i] << 16) * inv_sc, ha, la);
          split_e4m3(__uint_as_float(wv[i] & 0xFFFF0000u) * inv_sc, hb, lb);
          const int sh = 16 * (i & 1);
          hw[i >> 1] |= (static_cast<uint32_t>(ha) | (static_cast<uint32_t>(hb) << 8)) << sh;
          lw[i >> 1] |= (static_cast<uint32_t>(la) | (static_cast<uint32_t>(lb) << 8)) << sh;
        }
      }
      *reinterpret_cast<uint4*>(hi_row + c) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(lo_row + c) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    if (scale && tid == 0) *scale = sc;
  }
  __syncthreads();  // s_max is reused by the next row
}

}  // namespace fp8q
}  // namespace moe
