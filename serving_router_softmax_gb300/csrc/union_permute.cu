// moe_union_permute: the expert union of the verify tokens and the per-expert
// token groups.
//
// EcoSpec write-up, section 2: the experts a verify step must load in layer l
// are the union over verify tokens of the experts each token routes to.  The
// S2-MoE write-up (challenge 2) measures reuse as |union| / (s * k).
//
// Design: a single CTA.  A token-by-expert membership bitmap in shared memory
// (atomicOr, which also detects duplicate ids) gives both the union (a
// column-wise OR, scanned by one warp over <= 1024 experts) and each pair's
// rank inside its expert group (popcount of the expert's column over earlier
// tokens), so the permutation is deterministic and needs no sort.
#include "common.cuh"
#include "union_dev.cuh"

namespace moe {
namespace {

constexpr int kMaxE = unions::kMaxE;
constexpr int kMaxWords = 32768;  // T * ceil(E/32) bitmap words (128 KB)

__global__ void __launch_bounds__(1024) union_kernel(const int32_t* __restrict__ ids, int T, int k,
                                                     int E, int32_t* __restrict__ n_unique,
                                                     int32_t* __restrict__ unique,
                                                     int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ perm_token,
                                                     int32_t* __restrict__ perm_slot,
                                                     int32_t* __restrict__ inv,
                                                     float* __restrict__ reuse_ratio,
                                                     int32_t* dev_err) {
  extern __shared__ uint32_t member[];  // [T][EW]
  __shared__ unions::UnionSmem us;
  unions::union_block(ids, T, k, E, member, unions::view_of(us), n_unique, unique, offsets, perm_token, perm_slot, inv,
                      reuse_ratio, dev_err);
}

}  // namespace

int union_validate(int T, int k, int E) {
  if (T < 0 || k < 1 || k > 16 || E < 1 || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k > 65536) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * ((E + 31) / 32) > kMaxWords) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int union_launch(const int32_t* ids, int T, int k, int E, int32_t* n_unique, int32_t* unique,
                 int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, int32_t* inv,
                 float* reuse_ratio, int32_t* dev_err, cudaStream_t s) {
  size_t smem = static_cast<size_t>(T) * ((E + 31) / 32) * sizeof(uint32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxWords * static_cast<int>(sizeof(uint32_t))) != cudaSuccess)
    return MOE_ERR_CUDA;
  LaunchScope ls(kProfUnion, s);
  union_kernel<<<1, 1024, smem, s>>>(ids, T, k, E, n_unique, unique, offsets, perm_token, perm_slot,
                                     inv, reuse_ratio, dev_err);
  return check_launch();
}

}  // namespace moe

extern "C" int moe_union_permute(const int32_t* ids, int32_t T, int32_t k, int32_t E,
                                 int32_t* n_unique, int32_t* unique, int32_t* offsets,
                                 int32_t* perm_token, int32_t* perm_slot, int32_t* inv,
                                 float* reuse_ratio, int32_t* dev_err, void* stream) {
  int st = moe::union_validate(T, k, E);
  if (st != MOE_OK) return st;
  if (!n_unique || !unique || !offsets || !reuse_ratio) return MOE_ERR_ARG;
  if (T > 0 && (!ids || !perm_token || !perm_slot || !inv)) return MOE_ERR_ARG;
  return moe::union_launch(ids, T, k, E, n_unique, unique, offsets, perm_token, perm_slot, inv,
                           reuse_ratio, dev_err, static_cast<cudaStream_t>(stream));
}
