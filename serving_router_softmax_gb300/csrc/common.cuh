// Shared device/host helpers of libmoeverify (internal header).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/moe_verify.h"

namespace moe {

constexpr int kWarp = 32;

// Host-side launch bookkeeping (launch counter + optional event timing).
void note_launch(int cls, cudaStream_t s, bool before);
struct LaunchScope {
  int cls;
  cudaStream_t s;
  LaunchScope(int c, cudaStream_t st) : cls(c), s(st) { note_launch(cls, s, true); }
  ~LaunchScope() { note_launch(cls, s, false); }
};

enum ProfClass { kProfEco = 0, kProfRoute = 1, kProfUnion = 2, kProfPrep = 3, kProfGateUp = 4,
                 kProfDown = 5, kProfCombine = 6, kProfRouter = 7, kProfS2 = 8, kProfStage = 9,
                 kProfHot = 10, kProfDepth = 11 };

int sm_count();
// Test-hook bits set by moe_test_set_stall (0 in normal operation).
int test_stall_mask();

// NVTX range around a host-side span (a step's or plan's enqueue, one of
// their layers), pushed only while moe_set_nvtx(1) is in effect.
struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name);
  ~NvtxRange();
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

inline int check_launch() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Launches `kernel`, optionally with programmatic dependent launch: the
// kernel may start before its predecessor in the stream finishes and must
// execute griddepcontrol.wait before touching anything the predecessor writes
// or reads.  Every kernel of this library that is launched this way does so.
template <typename... KArgs, typename... Args>
int launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Grid-dependency control (no-ops for kernels launched without PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Store with release semantics at GPU scope: writes this thread made, or
// observed through a barrier, before it are visible to a reader that
// acquires the stored value.
__device__ __forceinline__ void st_release_gpu(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void flag_error(int32_t* dev_err, int32_t bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// Inclusive prefix sums over the 32 lanes of a fully populated warp (every
// lane calls it).  Unrolled and branch-free: the lane test is a select, so no
// lane diverges between the shuffles.  The same scan written as a rolled loop
// around an `if (lane >= off)` measured about 600 SM cycles per step on GB300
// against about 50 for this form.
__device__ __forceinline__ int warp_inclusive_sum(int v, int lane) {
  __syncwarp();
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, v, off);
    v += lane >= off ? a : 0;
  }
  return v;
}

__device__ __forceinline__ void warp_inclusive_sum2(int& v, int& w, int lane) {
  __syncwarp();
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, v, off);
    const int b = __shfl_up_sync(0xFFFFFFFFu, w, off);
    v += lane >= off ? a : 0;
    w += lane >= off ? b : 0;
  }
}

// Total order used by every top-k: larger value first, equal values -> lower id.
__device__ __forceinline__ bool topk_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits_rn(float f) {
  // Round to nearest even; inputs here are finite.
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Expert slots held by a layer's weight buffers, and the expert -> slot table
// (NULL when every expert sits at its own index).
inline int weight_slots(const moe_layer_weights& lw) { return lw.pool ? lw.pool->n_slots : lw.E; }
inline const int32_t* slot_table(const moe_layer_weights& lw) { return lw.pool ? lw.pool->slot_of : nullptr; }

// Slot of expert e (a valid id) in the weight buffers, -1 if the table holds
// a value outside [0, n_slots).
__device__ __forceinline__ int weight_slot(const int32_t* slot_of, int n_slots, int e) {
  if (!slot_of) return e;
  const int s = slot_of[e];
  return s >= 0 && s < n_slots ? s : -1;
}

// The next layer's predicted experts, prefetched into L2 by the tensor-core
// down kernels of the whole step once each CTA has issued its last weight
// load: HBM is underused from the end of a down launch until the next
// layer's gate/up stream starts.  The predicted experts are the set bits
// [bit0, bit0 + E) of the OR of `rows` rows of pred_B (W words each: the
// selection's final expert buffers); expert e's gate/up weights are the
// bytes [e * expert_bytes, (e + 1) * expert_bytes) of base (tiled layout,
// resident weights).  `budget` bytes over the whole grid, split evenly over
// the predicted experts from the start of each one's weights.
struct NextLayerPrefetch {
  const uint8_t* base;  // NULL: no prefetch
  long long expert_bytes;
  long long budget;
  const uint32_t* pred_B;
  int32_t rows, W, bit0;
};

// Host-side FFN internals shared by the standalone call and the whole step.
struct FfnArgs {
  const void* x;            // [*, H] activations (fp32 or bf16 bits)
  const int32_t* x_rows;    // optional row map: token t uses row x_rows[t] of x
  int32_t x_rows_limit;     // rows of x (bound for x_rows)
  int32_t T, k;
  moe_layer_weights lw;
  const int32_t* n_unique;
  const int32_t* unique;
  const int32_t* offsets;
  const int32_t* perm_token;
  const int32_t* inv;
  const float* w;
  float* y;
  void* ws;
  size_t ws_bytes;
  int32_t* dev_err;
  cudaStream_t stream;
  bool pdl_first;           // the first FFN kernel may start before the caller's previous kernel ends
  // Whole step, bf16 tensor-core layers with T <= 32 and resident weights:
  // the layer-head kernel already copied the token rows and zeroed the
  // fix-up counters (no prep kernel), and publishes ready_value in
  // ready_flag once the union is written (see TcParams::ready_flag).
  bool head_prepared;
  int32_t* ready_flag;
  int32_t ready_value;
  // Whole step, tensor-core layers: the next layer's predicted experts,
  // which the down CTAs ask L2 to fetch after their last weight load.
  NextLayerPrefetch pf;
};
size_t ffn_workspace_bytes(const moe_layer_weights& lw, int T, int k);
int ffn_validate(const moe_layer_weights& lw, int T, int k);
int ffn_launch(const FfnArgs& a);

// Work of the bf16 tensor-core FFN's prep kernel that the layer-head kernel
// can take over (token-dense layers, T <= 32, resident weights): copy the T
// token rows of x (through the row map) into xd and zero n_counters fix-up
// counters.  The head then also publishes the union to the gate/up kernel
// through ready_flag.  ffn_head_prep returns false when the layer does not
// qualify; the pointers lie in the FFN workspace `ws`.
struct HeadPrep {
  const uint16_t* x;        // [rows, H] bf16 bits
  const int32_t* x_rows;    // token t uses row x_rows[t]
  int32_t x_rows_limit;
  int32_t H;
  uint16_t* xd;             // [T, H]
  int32_t* counters;
  int32_t n_counters;
  int32_t* ready_flag;      // written ready_value (release) once the union is out
  int32_t ready_value;
  // FP8 layers: the token rows are quantized (hi/lo E4M3 rows of xq_hi /
  // xq_lo with one power-of-two scale per row in xscale) instead of copied
  // to xd; rows T..q_rows-1 get scale 1.  NULL for bf16 layers.
  uint8_t* xq_hi;
  uint8_t* xq_lo;
  float* xscale;
  int32_t q_rows;
};
bool ffn_head_prep(const moe_layer_weights& lw, int T, int k, void* ws, HeadPrep* hp);

// Expert staging (layers with an expert pool).
bool expert_bytes(const moe_layer_weights& lw, size_t* gate_up, size_t* down);
int stage_validate(const moe_layer_weights& lw);
int stage_launch(const moe_layer_weights& lw, const int32_t* n_unique, const int32_t* unique, int32_t* n_staged,
                 int32_t* dev_err, cudaStream_t s, bool pdl);

// Route internals (optional row map into a node table, optional confidence map).
struct RouteArgs {
  const float* logits;      // [*, E]
  const int32_t* rows;      // optional: token t uses logits row rows[t]
  int32_t rows_limit;       // rows of logits (bound for rows)
  const float* w_conf;      // [T] or NULL
  moe_route_cfg cfg;
  int32_t* ids;
  float* w;
  int32_t* dev_err;
  cudaStream_t stream;
};
int route_validate(const moe_route_cfg& c, bool have_conf);
int route_launch(const RouteArgs& a);

int union_validate(int T, int k, int E);

// Fused route + union for one layer of the whole step (single CTA).
// rows_ready: the row map was complete before the launch (it may be read
// before the wait on the previous kernel).
// hp (optional): the FFN prep work and union handshake of HeadPrep, done by
// extra CTAs of the same launch (CTA 0 routes).
int layer_head_launch(const RouteArgs& ra, int32_t* n_unique, int32_t* unique, int32_t* offsets,
                      int32_t* perm_token, int32_t* perm_slot, int32_t* inv, float* reuse_ratio, bool pdl,
                      bool rows_ready, const HeadPrep* hp = nullptr);
int union_launch(const int32_t* ids, int T, int k, int E, int32_t* n_unique, int32_t* unique,
                 int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, int32_t* inv,
                 float* reuse_ratio, int32_t* dev_err, cudaStream_t s);

// Router logits (optionally launched with programmatic dependent launch).
struct RouterArgs {
  const void* x;            // [T, H] fp32 or bf16 bits
  const void* w_router;     // [E, H] fp32 or bf16 bits
  moe_router_cfg cfg;
  float* logits;            // [T, E]
  cudaStream_t stream;
  bool pdl;
};
int router_validate(const moe_router_cfg& c);
int router_launch(const RouterArgs& a);

struct EcoArgs {
  const float* P;
  const int32_t* parent;
  const uint32_t* own_fp;
  int32_t nseq;
  const int32_t* gamma;
  eco_cfg cfg;
  int32_t* selected;
  int32_t* union_size;
  int32_t* dev_err;
  // Optional outputs for the whole step: verify token rows into the
  // [nseq, N+1] node table and the token confidences (path probabilities).
  int32_t* verify_rows;
  float* verify_conf;
  int32_t T_expected;
  cudaStream_t stream;
  // Whole step: the FFN's union-ready word, cleared here at the start of
  // every step (so that a value left by an interrupted step is never taken
  // for a fresh one).  NULL: nothing to clear.
  int32_t* ready_flag;
  // Optional: the final expert buffer B of each sequence ([nseq][W] words;
  // one buffer for the whole batch in mode 2, written to row 0 with the
  // other rows zero): the predicted (layer, expert) union of the verify
  // tokens other than the roots.
  uint32_t* pred_B;
};
int eco_validate(const eco_cfg& c, int nseq);
int eco_launch(const EcoArgs& a);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace moe
