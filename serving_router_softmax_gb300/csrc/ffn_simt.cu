// moe_verify_ffn, CUDA-core path: grouped SwiGLU expert FFN over the expert
// union, plus the weighted combine.
//
// EcoSpec write-up, section 1: a verify step's MoE cost is the union of
// experts its tokens activate, so each unique expert's weights are streamed
// once and applied to every token routed to it.  FFN_e(x) =
// W_down (silu(W_gate x) * (W_up x)); y_t = sum_j w_tj FFN_{e(t,j)}(x_t).
//
// This path serves fp32 weights (the 1e-4 tolerance of the fp32 workload rules
// out TF32 tensor cores) and is the reference-free fallback for the other
// dtypes.  Work item = one output row of one unique expert; a warp streams
// that weight row with 16-byte loads, applies it to up to 8 of the expert's
// tokens per pass, and reduces with shuffles.  The grid is sized from the
// device-side union size by a grid-stride loop, so no host sync is needed.
#include <cuda_fp8.h>

#include "common.cuh"
#include "ffn_internal.cuh"

namespace moe {
namespace {

constexpr int kTokChunk = 8;

template <int DT>
struct Vec;  // elements per 16-byte vector and their decode
template <>
struct Vec<MOE_DTYPE_F32> {
  static constexpr int N = 4;
  __device__ static void load(const void* p, float* out) {
    float4 v = *reinterpret_cast<const float4*>(p);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  }
};
template <>
struct Vec<MOE_DTYPE_BF16> {
  static constexpr int N = 8;
  __device__ static void load(const void* p, float* out) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec<MOE_DTYPE_E4M3_B128> {
  static constexpr int N = 16;
  __device__ static void load(const void* p, float* out) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>(w[i] >> (16 * h));
        __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
        float2 f = __half22float2(*reinterpret_cast<__half2*>(&hr));
        out[4 * i + 2 * h] = f.x;
        out[4 * i + 2 * h + 1] = f.y;
      }
    }
  }
};

// Activations: fp32 for the fp32 dtype, bf16 otherwise.
template <int DT>
struct Act {
  static constexpr bool kF32 = DT == MOE_DTYPE_F32;
  // Loads `n` consecutive activations (n = 4, 8 or 16; 16-byte aligned groups).
  template <int NV>
  __device__ static void load(const void* base, size_t idx, float* out) {
    if (kF32) {
      const float* p = reinterpret_cast<const float*>(base) + idx;
#pragma unroll
      for (int i = 0; i < NV; i += 4) {
        float4 v = *reinterpret_cast<const float4*>(p + i);
        out[i] = v.x; out[i + 1] = v.y; out[i + 2] = v.z; out[i + 3] = v.w;
      }
    } else {
      const uint16_t* p = reinterpret_cast<const uint16_t*>(base) + idx;
#pragma unroll
      for (int i = 0; i < NV; i += 8) {
        uint4 v = *reinterpret_cast<const uint4*>(p + i);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          out[i + 2 * q] = __uint_as_float(w[q] << 16);
          out[i + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
        }
      }
    }
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

__device__ __forceinline__ float silu_mul(float a, float b) { return a / (1.f + expf(-a)) * b; }

// Checks the union produced by moe_union_permute before it is used to index
// memory; returns U, or -1 (after flagging) if it is out of range.
__device__ __forceinline__ int checked_union_size(const int32_t* n_unique, int cap, int32_t* dev_err) {
  int U = *n_unique;
  if (U < 0 || U > cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(dev_err, MOE_DEV_CAPACITY);
    return -1;
  }
  return U;
}

template <int DT>
__global__ void __launch_bounds__(256) gateup_simt_kernel(
    const void* __restrict__ x, const int32_t* __restrict__ x_rows, int x_rows_limit, int T, int k,
    int H, int I, int E, const void* __restrict__ wgu, const float* __restrict__ sgu,
    const int32_t* __restrict__ slot_of, int n_slots,
    const int32_t* __restrict__ n_unique, const int32_t* __restrict__ unique,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm_token, void* __restrict__ h,
    int32_t* dev_err) {
  using V = Vec<DT>;
  constexpr int NV = V::N;
  constexpr int EB = DT == MOE_DTYPE_F32 ? 4 : (DT == MOE_DTYPE_BF16 ? 2 : 1);
  const int TK = T * k;
  const int U = checked_union_size(n_unique, min(E, TK), dev_err);
  if (U <= 0) return;
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (gridDim.x * (long long)blockDim.x) >> 5;
  const long long items = (long long)U * I;
  const int HB = H / 128;
  for (long long it = warp; it < items; it += nwarps) {
    const int u = static_cast<int>(it / I);
    const int i = static_cast<int>(it - (long long)u * I);
    const int e = unique[u];
    const int o0 = offsets[u], o1 = offsets[u + 1];
    const int ws = e >= 0 && e < E ? weight_slot(slot_of, n_slots, e) : -1;
    if (ws < 0 || o0 < 0 || o1 > TK || o0 > o1) {
      if (lane == 0) flag_error(dev_err, MOE_DEV_BAD_ID);
      continue;
    }
    const char* grow = reinterpret_cast<const char*>(wgu) + ((size_t)ws * 2 * I + i) * H * EB;
    const char* urow = grow + (size_t)I * H * EB;
    for (int c0 = o0; c0 < o1; c0 += kTokChunk) {
      const int nt = min(kTokChunk, o1 - c0);
      size_t xoff[kTokChunk];
      bool ok = true;
#pragma unroll
      for (int n = 0; n < kTokChunk; ++n) {
        int tok = n < nt ? perm_token[c0 + n] : 0;
        const bool tok_ok = tok >= 0 && tok < T;
        int row = (x_rows && n < nt && tok_ok) ? x_rows[tok] : tok;
        ok &= tok_ok && (!x_rows || (row >= 0 && row < x_rows_limit));
        xoff[n] = ok ? (size_t)row * H : 0;
      }
      if (!ok) {
        if (lane == 0) flag_error(dev_err, MOE_DEV_BAD_ID);
        continue;
      }
      float ag[kTokChunk], au[kTokChunk];
#pragma unroll
      for (int n = 0; n < kTokChunk; ++n) ag[n] = au[n] = 0.f;
      for (int kk = lane * NV; kk < H; kk += 32 * NV) {
        float gv[NV], uv[NV];
        V::load(grow + (size_t)kk * EB, gv);
        V::load(urow + (size_t)kk * EB, uv);
        float sg = 1.f, su = 1.f;
        if (DT == MOE_DTYPE_E4M3_B128) {
          const float* se = sgu + (size_t)e * (2 * I / 128) * HB;
          sg = se[(i / 128) * HB + kk / 128];
          su = se[((I + i) / 128) * HB + kk / 128];
        }
#pragma unroll
        for (int n = 0; n < kTokChunk; ++n) {
          if (n < nt) {
            float xv[NV];
            Act<DT>::template load<NV>(x, xoff[n] + kk, xv);
            float dg = 0.f, du = 0.f;
#pragma unroll
            for (int q = 0; q < NV; ++q) {
              dg = fmaf(gv[q], xv[q], dg);
              du = fmaf(uv[q], xv[q], du);
            }
            ag[n] = fmaf(sg, dg, ag[n]);
            au[n] = fmaf(su, du, au[n]);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < kTokChunk; ++n) {
        if (n < nt) {
          float a = warp_sum(ag[n]);
          float b = warp_sum(au[n]);
          if (lane == n) {
            float hv = silu_mul(a, b);
            size_t idx = (size_t)(c0 + n) * I + i;
            if (DT == MOE_DTYPE_F32)
              reinterpret_cast<float*>(h)[idx] = hv;
            else
              reinterpret_cast<uint16_t*>(h)[idx] = float_to_bf16_bits_rn(hv);
          }
        }
      }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(256) down_simt_kernel(
    int T, int k, int H, int I, int E, const void* __restrict__ wd, const float* __restrict__ sd,
    const int32_t* __restrict__ slot_of, int n_slots,
    const int32_t* __restrict__ n_unique, const int32_t* __restrict__ unique,
    const int32_t* __restrict__ offsets, const void* __restrict__ h, float* __restrict__ o,
    int32_t* dev_err) {
  using V = Vec<DT>;
  constexpr int NV = V::N;
  constexpr int EB = DT == MOE_DTYPE_F32 ? 4 : (DT == MOE_DTYPE_BF16 ? 2 : 1);
  // h is fp32 for the fp32 dtype and bf16 otherwise.
  constexpr int DTH = DT == MOE_DTYPE_F32 ? MOE_DTYPE_F32 : MOE_DTYPE_BF16;
  const int TK = T * k;
  const int U = checked_union_size(n_unique, min(E, TK), dev_err);
  if (U <= 0) return;
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (gridDim.x * (long long)blockDim.x) >> 5;
  const long long items = (long long)U * H;
  const int IB = I / 128;
  for (long long it = warp; it < items; it += nwarps) {
    const int u = static_cast<int>(it / H);
    const int r = static_cast<int>(it - (long long)u * H);
    const int e = unique[u];
    const int o0 = offsets[u], o1 = offsets[u + 1];
    const int ws = e >= 0 && e < E ? weight_slot(slot_of, n_slots, e) : -1;
    if (ws < 0 || o0 < 0 || o1 > TK || o0 > o1) {
      if (lane == 0) flag_error(dev_err, MOE_DEV_BAD_ID);
      continue;
    }
    const char* row = reinterpret_cast<const char*>(wd) + ((size_t)ws * H + r) * I * EB;
    for (int c0 = o0; c0 < o1; c0 += kTokChunk) {
      const int nt = min(kTokChunk, o1 - c0);
      float acc[kTokChunk];
#pragma unroll
      for (int n = 0; n < kTokChunk; ++n) acc[n] = 0.f;
      for (int kk = lane * NV; kk < I; kk += 32 * NV) {
        float wv[NV];
        V::load(row + (size_t)kk * EB, wv);
        float sc = 1.f;
        if (DT == MOE_DTYPE_E4M3_B128) sc = sd[((size_t)e * (H / 128) + r / 128) * IB + kk / 128];
#pragma unroll
        for (int n = 0; n < kTokChunk; ++n) {
          if (n < nt) {
            float hv[NV];
            Act<DTH>::template load<NV>(h, (size_t)(c0 + n) * I + kk, hv);
            float d = 0.f;
#pragma unroll
            for (int q = 0; q < NV; ++q) d = fmaf(wv[q], hv[q], d);
            acc[n] = fmaf(sc, d, acc[n]);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < kTokChunk; ++n) {
        if (n < nt) {
          float v = warp_sum(acc[n]);
          if (lane == n) o[(size_t)(c0 + n) * H + r] = v;
        }
      }
    }
  }
}

}  // namespace

// y[t, :] = sum_j w[t, j] * o[inv[t*k + j], :], slots in order.  Shared by
// all FFN paths; after the tensor-core down kernels it is launched with
// programmatic dependent launch.
constexpr int kCombK = 16;  // largest k (checked by ffn_validate)

__global__ void __launch_bounds__(256) combine_kernel(int T, int k, int H, int E,
                                                      const int32_t* __restrict__ n_unique,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w,
                                                      const float* __restrict__ o,
                                                      float* __restrict__ y, int32_t* dev_err) {
  const int TK = T * k;
  const long long total = (long long)T * (H / 4);
  const long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // All of an item's slot indices and weights, then all of its rows of o,
  // are requested before the first use, so the loads overlap; the sum still
  // runs in slot order.  The union size, indices and weights come from the
  // routing kernels, which finished before the down projection this kernel
  // follows started (only o is that kernel's result), so the first item's
  // are read before the wait.
  int pj[kCombK];
  float wj[kCombK];
  auto load_slots = [&](long long i) {
    const int t = static_cast<int>(i / (H / 4));
#pragma unroll
    for (int j = 0; j < kCombK; ++j) {
      pj[j] = -1;
      wj[j] = 0.f;
      if (j < k) {
        pj[j] = inv[t * k + j];
        wj[j] = w[t * k + j];
      }
    }
  };
  const int U = *n_unique;
  const bool valid = U > 0 && U <= min(E, TK);
  if (valid && i0 < total) load_slots(i0);
  pdl_wait();
  pdl_trigger();
  for (long long i = i0; i < total; i += stride) {
    const int t = static_cast<int>(i / (H / 4));
    const int c = static_cast<int>(i - (long long)t * (H / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      if (i != i0) load_slots(i);
      float4 v[kCombK];
#pragma unroll
      for (int j = 0; j < kCombK; ++j) {
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < k && pj[j] >= 0 && pj[j] < TK) v[j] = *reinterpret_cast<const float4*>(o + (size_t)pj[j] * H + c);
      }
#pragma unroll
      for (int j = 0; j < kCombK; ++j) {
        if (j >= k) break;
        if (pj[j] < 0 || pj[j] >= TK) {
          flag_error(dev_err, MOE_DEV_BAD_ID);
          continue;
        }
        acc.x = fmaf(wj[j], v[j].x, acc.x);
        acc.y = fmaf(wj[j], v[j].y, acc.y);
        acc.z = fmaf(wj[j], v[j].z, acc.z);
        acc.w = fmaf(wj[j], v[j].w, acc.w);
      }
    }
    *reinterpret_cast<float4*>(y + (size_t)t * H + c) = acc;
  }
}

int ffn_simt_launch(const FfnArgs& a, const FfnWorkspace& ws) {
  const auto& lw = a.lw;
  const int sms = sm_count();
  const int blocks = sms * 8;
  cudaStream_t s = a.stream;
  switch (lw.dtype) {
#define MOE_SIMT_CASE(DT)                                                                              \
  case DT: {                                                                                          \
    {                                                                                                 \
      LaunchScope ls(kProfGateUp, s);                                                                 \
      gateup_simt_kernel<DT><<<blocks, 256, 0, s>>>(a.x, a.x_rows, a.x_rows_limit, a.T, a.k, lw.H,     \
                                                    lw.I, lw.E, lw.w_gate_up, lw.scales_gate_up,      \
                                                    slot_table(lw), weight_slots(lw),                 \
                                                    a.n_unique, a.unique, a.offsets, a.perm_token,    \
                                                    ws.h, a.dev_err);                                 \
    }                                                                                                 \
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;                                                \
    {                                                                                                 \
      LaunchScope ls(kProfDown, s);                                                                   \
      down_simt_kernel<DT><<<blocks, 256, 0, s>>>(a.T, a.k, lw.H, lw.I, lw.E, lw.w_down,              \
                                                  lw.scales_down, slot_table(lw), weight_slots(lw),   \
                                                  a.n_unique, a.unique, a.offsets,                    \
                                                  ws.h, ws.o, a.dev_err);                             \
    }                                                                                                 \
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;                                                \
    break;                                                                                            \
  }
    MOE_SIMT_CASE(MOE_DTYPE_F32)
    MOE_SIMT_CASE(MOE_DTYPE_BF16)
    MOE_SIMT_CASE(MOE_DTYPE_E4M3_B128)
#undef MOE_SIMT_CASE
    default:
      return MOE_ERR_UNSUPPORTED;
  }
  return combine_launch(a, ws.o, false);
}

int combine_launch(const FfnArgs& a, const float* o, bool pdl) {
  const int H = a.lw.H;
  long long total = (long long)a.T * (H / 4);
  int blocks = static_cast<int>((total + 255) / 256);
  int cap = sm_count() * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  LaunchScope ls(kProfCombine, a.stream);
  return launch_k(combine_kernel, dim3(blocks), dim3(256), 0, a.stream, pdl, a.T, a.k, H, a.lw.E, a.n_unique,
                  a.inv, a.w, o, a.y, a.dev_err);
}

}  // namespace moe
