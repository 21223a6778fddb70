// Device fill for the synthetic expert weights.
//
// Same definition as workload/counter_hash.py: element i of a stream with key K
// is derived from mix64(K + (i + 1) * GOLDEN), the SplitMix64 finaliser of
// Steele, Lea and Flood (OOPSLA 2014) used in counter mode.  This file is part
// of the input generator, not of the verify path: it only writes inputs.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kMix1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kMix2 = 0x94D049BB133111EBull;
constexpr int kScaleExp = 13;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * kMix1;
  z = (z ^ (z >> 27)) * kMix2;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t hash_at(uint64_t key, uint64_t idx) {
  return mix64(key + (idx + 1ull) * kGolden);
}

__device__ __forceinline__ float grid8(uint64_t h) {
  int b = static_cast<int>(h >> 56);
  return static_cast<float>(2 * b - 255) * 0x1p-13f;
}

__device__ __forceinline__ uint8_t e4m3_code(uint64_t h) {
  uint8_t c = static_cast<uint8_t>(h >> 56);
  if ((c & 0x7F) == 0x7F) c ^= 1;
  return c;
}

__device__ __forceinline__ float scale_val(uint64_t h) {
  uint32_t f = static_cast<uint32_t>((h >> 33) & 0x7FFFFFull);
  // 1 + f * 2^-23 is exact in fp32; the power-of-two factor is exact too.
  float m = __uint_as_float(0x3F800000u | f);
  return ldexpf(m, -kScaleExp);
}

// kind 0: bf16 grid8, 1: fp32 grid8, 2: e4m3 codes, 3: fp32 scales.
// Each thread writes 8 consecutive elements; full groups of 8 are stored with
// vector stores (dst is a fresh allocation, so 16-byte aligned), the ragged end
// element by element.
__global__ void fill_kernel(void* dst, int kind, uint64_t n, uint64_t key, uint64_t idx0) {
  uint64_t t = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x;
  uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t base = t * 8; base < n; base += stride * 8) {
    uint64_t cnt = (n - base) < 8 ? (n - base) : 8;
    uint32_t w[8];
    for (uint64_t j = 0; j < 8; ++j) {
      uint64_t h = hash_at(key, idx0 + base + j);
      if (kind == 0) w[j] = __float_as_uint(grid8(h)) >> 16;
      else if (kind == 1) w[j] = __float_as_uint(grid8(h));
      else if (kind == 2) w[j] = e4m3_code(h);
      else w[j] = __float_as_uint(scale_val(h));
    }
    if (cnt == 8) {
      if (kind == 0) {
        uint4 v = make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16), w[6] | (w[7] << 16));
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(dst) + base) = v;
      } else if (kind == 2) {
        uint2 v = make_uint2(w[0] | (w[1] << 8) | (w[2] << 16) | (w[3] << 24),
                             w[4] | (w[5] << 8) | (w[6] << 16) | (w[7] << 24));
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(dst) + base) = v;
      } else {
        uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<uint32_t*>(dst) + base);
        p[0] = make_uint4(w[0], w[1], w[2], w[3]);
        p[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
      for (uint64_t j = 0; j < cnt; ++j) {
        uint64_t i = base + j;
        if (kind == 0) reinterpret_cast<uint16_t*>(dst)[i] = static_cast<uint16_t>(w[j]);
        else if (kind == 2) reinterpret_cast<uint8_t*>(dst)[i] = static_cast<uint8_t>(w[j]);
        else reinterpret_cast<uint32_t*>(dst)[i] = w[j];
      }
    }
  }
}

}  // namespace

extern "C" int gen_fill(void* dst, int kind, uint64_t n, uint64_t key, uint64_t idx0, void* stream) {
  if (n == 0) return 0;
  if (dst == nullptr || kind < 0 || kind > 3) return 1;
  if (reinterpret_cast<uintptr_t>(dst) % 16 != 0) return 1;  // vector stores need 16-byte alignment
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 3;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t threads_needed = (n + 7) / 8;
  uint64_t blocks = (threads_needed + 255) / 256;
  uint64_t cap = static_cast<uint64_t>(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, kind, n, key, idx0);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
