// moe_pack_tiled: load-time repacking of one layer's expert weights into the
// tile-contiguous layout the tensor-core FFN streams best (include/moe_verify.h,
// MOE_LAYOUT_TILED).  A block covers 128 rows and 128 bytes of the reduction
// dimension (64 bf16 or 128 FP8 values); one thread per 16-byte vector of the
// destination; rows past the matrix end are written as zeros.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRowsPerTile = 128;
constexpr int kBlockBytes = 128;  // reduction bytes per block row (8 vectors)

// gate/up: block (e, m, kb) = [256][128 B]: rows 0..127 gate, 128..255 up.
// src rows are row_bytes long; I rows of gate then I rows of up per expert.
__global__ void pack_gate_up_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, long long row_bytes,
                                    int I, int E, int MT) {
  const int KB = static_cast<int>(row_bytes / kBlockBytes);
  const long long nvec = (long long)E * MT * KB * 256 * 8;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
       v += (long long)gridDim.x * blockDim.x) {
    const int vec = static_cast<int>(v & 7);
    const long long rowg = v >> 3;  // global packed row
    const int r = static_cast<int>(rowg % 256);
    const long long blk = rowg / 256;
    const int kb = static_cast<int>(blk % KB);
    const long long em = blk / KB;
    const int m = static_cast<int>(em % MT);
    const int e = static_cast<int>(em / MT);
    const int row = m * kRowsPerTile + (r & 127);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (row < I) {
      const long long srow = (long long)e * 2 * I + (r < 128 ? row : I + row);
      val = *reinterpret_cast<const uint4*>(src + srow * row_bytes + (long long)kb * kBlockBytes + vec * 16);
    }
    *reinterpret_cast<uint4*>(dst + v * 16) = val;
  }
}

// down: block (e, m, kb) = [128][128 B] of W_down rows m*128.., columns kb*128 B..
__global__ void pack_down_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, long long row_bytes,
                                 int H, int E, int MT) {
  const int KB = static_cast<int>(row_bytes / kBlockBytes);
  const long long nvec = (long long)E * MT * KB * 128 * 8;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
       v += (long long)gridDim.x * blockDim.x) {
    const int vec = static_cast<int>(v & 7);
    const long long rowg = v >> 3;
    const int r = static_cast<int>(rowg % 128);
    const long long blk = rowg / 128;
    const int kb = static_cast<int>(blk % KB);
    const long long em = blk / KB;
    const int m = static_cast<int>(em % MT);
    const int e = static_cast<int>(em / MT);
    const int row = m * kRowsPerTile + r;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (row < H)
      val = *reinterpret_cast<const uint4*>(src + ((long long)e * H + row) * row_bytes + (long long)kb * kBlockBytes +
                                            vec * 16);
    *reinterpret_cast<uint4*>(dst + v * 16) = val;
  }
}

int elem_bytes(int dtype) { return dtype == MOE_DTYPE_BF16 ? 2 : (dtype == MOE_DTYPE_E4M3_B128 ? 1 : 0); }

bool tiled_sizes(const moe_layer_weights& lw, size_t* gu, size_t* dn) {
  const int eb = elem_bytes(lw.dtype);
  if (eb == 0 || lw.E < 1 || lw.E > 1024) return false;
  const int mult = kBlockBytes / eb;  // reduction elements per block
  if (lw.H < mult || lw.I < mult || lw.H % mult || lw.I % mult) return false;
  const size_t MTg = (lw.I + 127) / 128, MTd = (lw.H + 127) / 128;
  *gu = static_cast<size_t>(lw.E) * MTg * 256 * static_cast<size_t>(lw.H) * eb;
  *dn = static_cast<size_t>(lw.E) * MTd * 128 * static_cast<size_t>(lw.I) * eb;
  return true;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_tiled_bytes(const moe_layer_weights* lw, size_t* gate_up_bytes, size_t* down_bytes) {
  size_t gu = 0, dn = 0;
  if (!lw || !moe::tiled_sizes(*lw, &gu, &dn)) return 0;
  if (gate_up_bytes) *gate_up_bytes = gu;
  if (down_bytes) *down_bytes = dn;
  return gu + dn;
}

extern "C" int moe_pack_tiled(const moe_layer_weights* src, void* dst_gate_up, void* dst_down, void* stream) {
  using namespace moe;
  if (!src || src->layout != MOE_LAYOUT_ROWMAJOR || src->pool) return MOE_ERR_ARG;
  size_t gu = 0, dn = 0;
  if (!tiled_sizes(*src, &gu, &dn)) return MOE_ERR_UNSUPPORTED;
  if (!src->w_gate_up || !src->w_down || !dst_gate_up || !dst_down) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(src->w_gate_up) | reinterpret_cast<uintptr_t>(src->w_down) |
       reinterpret_cast<uintptr_t>(dst_gate_up) | reinterpret_cast<uintptr_t>(dst_down)) & 15)
    return MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = sm_count() * 8;
  const int eb = elem_bytes(src->dtype);
  const int MTg = (src->I + 127) / 128, MTd = (src->H + 127) / 128;
  pack_gate_up_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(src->w_gate_up),
                                             static_cast<uint8_t*>(dst_gate_up), (long long)src->H * eb, src->I,
                                             src->E, MTg);
  if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
  pack_down_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(src->w_down),
                                          static_cast<uint8_t*>(dst_down), (long long)src->I * eb, src->H, src->E,
                                          MTd);
  return check_launch();
}
