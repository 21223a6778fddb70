// moe_stage_experts: expert-level residency on a Grace-Blackwell node.
//
// S2-MoE write-up, "system implementation: expert-level offloading": the
// non-expert parameters and a profiled list of frequently activated (hot)
// experts stay in device memory; any other expert is fetched on demand.  On
// GB300 the cold experts sit in the Grace memory, which the GPU reads directly
// over NVLink-C2C.  The layer's union is only known on the device, so the
// fetch is a kernel: it lists the union's cold experts in union order, gives
// the c-th of them staging slot stage_first + c, records every union
// expert's slot in slot_of and copies the cold experts' weights into their
// slots.  The FFN then reads every expert of the union from HBM through
// slot_of; no host round trip sits between routing and the FFN.
//
// The copy is SM-driven: every thread keeps kUnroll 16-byte loads of host
// memory in flight before it stores them, so the whole grid holds several MB
// of outstanding reads, enough to cover the link's latency.  No bulk-tensor
// (TMA) copy touches host memory.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kStageThreads = 256;
constexpr int kUnroll = 8;
constexpr long long kChunk = static_cast<long long>(kStageThreads) * kUnroll * 16;  // 32 KB per CTA pass
constexpr int kMaxUnion = 1024;  // E <= 1024

struct StageArgs {
  int E, n_slots, stage_first, n_stage;
  const int32_t* n_unique;
  const int32_t* unique;
  const int32_t* home_slot;
  const uint8_t* host_gu;
  const uint8_t* host_dn;
  uint8_t* pool_gu;
  uint8_t* pool_dn;
  long long gu_bytes, dn_bytes;   // one expert
  long long gu_chunks, dn_chunks; // kChunk pieces of one expert
  int32_t* slot_of;
  int32_t* n_staged;
  int32_t* dev_err;
};

__global__ void __launch_bounds__(kStageThreads) stage_kernel(const StageArgs a) {
  __shared__ int32_t cold_e[kMaxUnion];  // cold experts of the union, union order
  __shared__ int32_t warp_cnt[kStageThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool lead = blockIdx.x == 0;
  int U = *a.n_unique;
  if (U < 0 || U > a.E) {
    if (lead && tid == 0) flag_error(a.dev_err, MOE_DEV_CAPACITY);
    U = 0;
  }
  // Every CTA lists the cold experts (at most E <= 1024 reads); CTA 0 also
  // writes the slot table.
  int n_cold = 0;  // uniform across the CTA
  for (int u0 = 0; u0 < U; u0 += kStageThreads) {
    const int u = u0 + tid;
    int e = -1, h = -1;
    bool cold = false, bad = false;
    if (u < U) {
      e = a.unique[u];
      if (e < 0 || e >= a.E) {
        bad = true;
      } else {
        h = a.home_slot[e];
        cold = h == -1;
        bad = !cold && (h < 0 || h >= a.n_slots || (h >= a.stage_first && h < a.stage_first + a.n_stage));
      }
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, cold);
    if (lane == 0) warp_cnt[wid] = __popc(m);
    __syncthreads();
    int c = n_cold + __popc(m & ((1u << lane) - 1u)), tot = 0;
    for (int w2 = 0; w2 < kStageThreads / 32; ++w2) {
      if (w2 < wid) c += warp_cnt[w2];
      tot += warp_cnt[w2];
    }
    if (cold && c < a.n_stage) cold_e[c] = e;
    if (lead && u < U) {
      if (bad) flag_error(a.dev_err, MOE_DEV_BAD_ID);
      if (cold && c >= a.n_stage) flag_error(a.dev_err, MOE_DEV_CAPACITY);
      if (e >= 0 && e < a.E) a.slot_of[e] = bad ? -1 : (cold ? (c < a.n_stage ? a.stage_first + c : -1) : h);
    }
    n_cold += tot;
    __syncthreads();
  }
  const int n_copy = n_cold < a.n_stage ? n_cold : a.n_stage;
  if (lead && tid == 0 && a.n_staged) *a.n_staged = n_copy;

  // Copy: work item i = (cold expert c, chunk r of its gate/up then down bytes).
  const long long per = a.gu_chunks + a.dn_chunks;
  const long long total = static_cast<long long>(n_copy) * per;
  for (long long i = blockIdx.x; i < total; i += gridDim.x) {
    const int c = static_cast<int>(i / per);
    const long long r = i - static_cast<long long>(c) * per;
    const long long e = cold_e[c];
    const long long slot = a.stage_first + c;
    const uint4* src;
    uint4* dst;
    long long len;
    if (r < a.gu_chunks) {
      const long long off = r * kChunk;
      src = reinterpret_cast<const uint4*>(a.host_gu + e * a.gu_bytes + off);
      dst = reinterpret_cast<uint4*>(a.pool_gu + slot * a.gu_bytes + off);
      len = a.gu_bytes - off < kChunk ? a.gu_bytes - off : kChunk;
    } else {
      const long long off = (r - a.gu_chunks) * kChunk;
      src = reinterpret_cast<const uint4*>(a.host_dn + e * a.dn_bytes + off);
      dst = reinterpret_cast<uint4*>(a.pool_dn + slot * a.dn_bytes + off);
      len = a.dn_bytes - off < kChunk ? a.dn_bytes - off : kChunk;
    }
    const int nv = static_cast<int>(len / 16);
    uint4 v[kUnroll];
    if (nv == kUnroll * kStageThreads) {
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) v[j] = __ldg(src + tid + j * kStageThreads);
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) dst[tid + j * kStageThreads] = v[j];
    } else {
      for (int idx = tid; idx < nv; idx += kStageThreads) dst[idx] = __ldg(src + idx);
    }
  }
}

}  // namespace

bool expert_bytes(const moe_layer_weights& lw, size_t* gu, size_t* dn) {
  const int eb = lw.dtype == MOE_DTYPE_F32 ? 4 : (lw.dtype == MOE_DTYPE_BF16 ? 2 : (lw.dtype == MOE_DTYPE_E4M3_B128 ? 1 : 0));
  if (eb == 0 || lw.H < 1 || lw.I < 1) return false;
  const size_t H = lw.H, I = lw.I;
  if (lw.layout == MOE_LAYOUT_TILED) {
    *gu = (I + 127) / 128 * 256 * H * eb;
    *dn = (H + 127) / 128 * 128 * I * eb;
  } else if (lw.layout == MOE_LAYOUT_ROWMAJOR) {
    *gu = 2 * I * H * eb;
    *dn = H * I * eb;
  } else {
    return false;
  }
  return true;
}

int stage_validate(const moe_layer_weights& lw) {
  int st = ffn_validate(lw, 1, 1);
  if (st != MOE_OK) return st;
  if (!lw.pool || !lw.pool->home_slot) return MOE_ERR_ARG;
  const moe_expert_pool& pl = *lw.pool;
  if (pl.n_stage > 0) {
    if (!pl.host_gate_up || !pl.host_down) return MOE_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(pl.host_gate_up) | reinterpret_cast<uintptr_t>(pl.host_down)) & 15)
      return MOE_ERR_ARG;
  }
  return MOE_OK;
}

int stage_launch(const moe_layer_weights& lw, const int32_t* n_unique, const int32_t* unique, int32_t* n_staged,
                 int32_t* dev_err, cudaStream_t s, bool pdl) {
  size_t gu = 0, dn = 0;
  if (!expert_bytes(lw, &gu, &dn)) return MOE_ERR_ARG;
  const moe_expert_pool& pl = *lw.pool;
  StageArgs a;
  a.E = lw.E;
  a.n_slots = pl.n_slots;
  a.stage_first = pl.stage_first;
  a.n_stage = pl.n_stage;
  a.n_unique = n_unique;
  a.unique = unique;
  a.home_slot = pl.home_slot;
  a.host_gu = static_cast<const uint8_t*>(pl.host_gate_up);
  a.host_dn = static_cast<const uint8_t*>(pl.host_down);
  a.pool_gu = static_cast<uint8_t*>(const_cast<void*>(lw.w_gate_up));
  a.pool_dn = static_cast<uint8_t*>(const_cast<void*>(lw.w_down));
  a.gu_bytes = static_cast<long long>(gu);
  a.dn_bytes = static_cast<long long>(dn);
  a.gu_chunks = (a.gu_bytes + kChunk - 1) / kChunk;
  a.dn_chunks = (a.dn_bytes + kChunk - 1) / kChunk;
  a.slot_of = pl.slot_of;
  a.n_staged = n_staged;
  a.dev_err = dev_err;
  LaunchScope ls(kProfStage, s);
  return launch_k(stage_kernel, dim3(sm_count() * 2), dim3(kStageThreads), 0, s, pdl, a);
}

}  // namespace moe

extern "C" size_t moe_expert_bytes(const moe_layer_weights* lw, size_t* gate_up_bytes, size_t* down_bytes) {
  size_t gu = 0, dn = 0;
  if (!lw || moe::ffn_validate(*lw, 1, 1) != MOE_OK || !moe::expert_bytes(*lw, &gu, &dn)) return 0;
  if (gate_up_bytes) *gate_up_bytes = gu;
  if (down_bytes) *down_bytes = dn;
  return gu + dn;
}

extern "C" int moe_stage_experts(const moe_layer_weights* lw, const int32_t* n_unique, const int32_t* unique,
                                 int32_t* n_staged, int32_t* dev_err, void* stream) {
  if (!lw) return MOE_ERR_ARG;
  int st = moe::stage_validate(*lw);
  if (st != MOE_OK) return st;
  if (!n_unique || !unique) return MOE_ERR_ARG;
  return moe::stage_launch(*lw, n_unique, unique, n_staged, dev_err, static_cast<cudaStream_t>(stream), false);
}
