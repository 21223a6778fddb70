/*
 * moe_verify.h -- C ABI of the MoE speculative-verify library (libmoeverify.so).
 *
 * The library computes the data-parallel hot path of one speculative-decoding
 * verify step of a Mixture-of-Experts model:
 *   eco_select         EcoSpec cost-aware greedy draft selection
 *   moe_router_logits  router (gate) logits x . W_r^T of the verify tokens
 *   moe_route          router top-k + softmax weights, optional S2-MoE reuse bias
 *   moe_union_permute  expert union of the verify tokens, per-expert token groups
 *   moe_verify_ffn     grouped SwiGLU expert FFN over the union + weighted combine
 *   moe_verify_step    all of the above for L layers in one call
 *   moe_verify_plan    the step's selection and per-layer routing/union only
 *   moe_stage_experts  copies a layer's cold experts of the union from host memory
 *   moe_hot_list       hot-expert list (and home-slot table) from profiled routing
 *   s2_expand          S2-MoE utility-driven draft expansion
 *   moe_depth_policy   confidence-gated depth per sequence (ragged speculation)
 *
 * Conventions shared by every entry point
 *   - Every array argument is a DEVICE pointer owned by the caller, unless a
 *     comment says "host".  The library never frees caller memory and keeps no
 *     pointer past the call.  The library allocates no device memory; kernels
 *     that need scratch space take a caller-provided workspace whose size the
 *     matching *_workspace() query returns.
 *   - `stream` is a cudaStream_t (passed as void*).  Every call only enqueues
 *     work on that stream and returns; it never synchronises the host.
 *   - The return value reports errors the host can see before launching
 *     (MOE_ERR_ARG for a bad size or NULL pointer, MOE_ERR_UNSUPPORTED for a
 *     shape outside the documented limits, MOE_ERR_CUDA for a launch failure,
 *     MOE_ERR_WORKSPACE for a too-small workspace).  Nothing is enqueued when a
 *     call returns an error.
 *   - Errors only the device can see (NaN logits, ids out of range, malformed
 *     trees, bounded waits that gave up) are OR-ed as MOE_DEV_* bits into
 *     `*dev_err` (an int32 in device memory that the caller zeroes and reads
 *     after synchronising).  Kernels never trap; when they flag an error they
 *     write the documented "invalid" values (-1 ids, zero counts) and return.
 *   - Arrays are row-major and densely packed.  Element types are as declared;
 *     bf16 tensors are passed as their 16-bit patterns, FP8 tensors as bytes.
 *   - Target: NVIDIA GB300 (sm_103a).  The library is built for that
 *     architecture only.
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_CUDA = 3,
  MOE_ERR_WORKSPACE = 4
};

/* Device error bits (OR-ed into *dev_err). */
#define MOE_DEV_NAN_LOGIT 0x01  /* a router logit was NaN: that token's ids are -1, weights 0  */
#define MOE_DEV_BAD_ID    0x02  /* an expert id outside [0, E)                                   */
#define MOE_DEV_DUP_ID    0x04  /* a token lists the same expert twice                           */
#define MOE_DEV_BAD_TREE  0x08  /* parent[t] not in [-1, t) or gamma outside [0, gamma_max]     */
#define MOE_DEV_BAD_PROB  0x10  /* a path probability / confidence weight is NaN or negative    */
#define MOE_DEV_TIMEOUT   0x20  /* a bounded device-side wait gave up                            */
#define MOE_DEV_CAPACITY  0x40  /* a count exceeded the capacity the caller sized buffers for   */
/* With an expert pool, an expert whose slot_of entry is outside [0, n_slots)
 * is reported by the FFN as MOE_DEV_BAD_ID; its weights are not read and the
 * outputs of the tokens routed to it are not valid. */

/* Weight storage types. */
enum {
  MOE_DTYPE_F32 = 0,       /* fp32 weights and activations                                  */
  MOE_DTYPE_BF16 = 1,      /* bf16 weights and activations                                  */
  MOE_DTYPE_E4M3_B128 = 2  /* FP8 E4M3 weights with one fp32 scale per 128x128 block;
                              bf16 activations                                              */
};

/* ---------------------------------------------------------------- router
 * moe_router_logits -- the gate's score of every expert for every token.
 *
 * Defined by: S2-MoE write-up, background (each MoE layer holds E expert
 * FFNs and a router/gate chooses each token's top-k of them) and EcoSpec
 * write-up section 2 (S_l(x_t), the experts token t routes to at layer l, is
 * a function of its hidden state x_t).  The gate is read as a bias-free
 * linear layer:
 *   logits[t, e] = sum_{h < H} x[t, h] * w_router[e, h]
 * with fp32 products and fp32 accumulation in a fixed order, so repeated
 * calls give identical bits.  The output is the input of moe_route.
 *
 *   x         [T, H] activations: cfg->x_dtype MOE_DTYPE_F32 or MOE_DTYPE_BF16
 *             (16-bit patterns).  16-byte aligned.
 *   w_router  [E, H] gate matrix: cfg->w_dtype MOE_DTYPE_F32 or
 *             MOE_DTYPE_BF16.  16-byte aligned.
 *   logits    [T, E] fp32 out.  4-byte aligned.
 * Limits: 8 <= H <= 1048576 with H % 8 == 0, 1 <= E <= 1024,
 * 0 <= T <= 65536 (T == 0 enqueues nothing and needs no pointers).
 * Errors: MOE_ERR_ARG for a negative size, a NULL or misaligned pointer;
 * MOE_ERR_UNSUPPORTED for sizes or dtypes outside the limits.  There are no
 * device-side errors: NaN or Inf inputs propagate into the logits, and
 * moe_route then flags MOE_DEV_NAN_LOGIT.
 * Accuracy: each logit carries at most 8 * ceil(H / 1024) + 8 roundings in
 * sequence, so |error| <= gamma_n * sum_h |x[t,h] * w_router[e,h]| with
 * n = 8 * ceil(H / 1024) + 8 and gamma_n = n u / (1 - n u), u = 2^-24.
 */
typedef struct {
  int32_t T, H, E;
  int32_t x_dtype, w_dtype;
} moe_router_cfg;

int moe_router_logits(const void* x, const void* w_router, const moe_router_cfg* cfg,
                      float* logits, void* stream);

/* ---------------------------------------------------------------- routing
 * moe_route -- per token: top-k experts of the router logits and their weights.
 *
 * Defined by: EcoSpec write-up section 3.1 (softmax, then top-K per layer) and
 * section 2 (S_l(x_t), the expert set token t routes to); with use_bias, the
 * S2-MoE write-up's component 2 (reuse-aware expert gating, steps 1-3, Fig. 5).
 *
 *   logits  [T, E] fp32.
 *   w_conf  [T] fp32 confidence weight per token (>= 0); read only when
 *           cfg->use_bias != 0, may be NULL otherwise.
 *   ids     [T, k] int32 out: expert ids in decreasing logit order; equal
 *           logits go to the lower id; -0.0 == +0.0.
 *   w       [T, k] fp32 out: softmax over the k selected logits (equal to the
 *           full softmax renormalised over the selected experts).
 * With use_bias the logits are first biased, in fp32 with this exact op order:
 *   g_e   = sum_{b = 0..T-1} w_conf[b] * [e in TopK(logits[b])]  (plain adds)
 *   E*    = the `cap` experts with the largest g_e among g_e > 0 (ties: lower id)
 *   lam_b = alpha * (logits[b]_(1) - logits[b]_(k+1))   ((j) = j-th largest)
 *   l'_b,e = logits[b,e] + lam_b for e in E*, unchanged otherwise
 * and ids/w are computed from l'.  Requires E >= k+1, cap >= 1.
 * Limits: 1 <= k <= 16, k <= E <= 1024, T >= 0; with use_bias T <= 256.
 * Device errors: MOE_DEV_NAN_LOGIT (token's ids = -1, w = 0),
 * MOE_DEV_BAD_PROB (w_conf NaN or negative; all ids -1).
 */
typedef struct {
  int32_t T, E, k;
  int32_t use_bias, cap;
  float alpha;
} moe_route_cfg;

int moe_route(const float* logits, const float* w_conf, const moe_route_cfg* cfg,
              int32_t* ids, float* w, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- union
 * moe_union_permute -- the experts the verify tokens need, each once.
 *
 * Defined by: EcoSpec write-up section 2 (the verify expert set is the union
 * of the tokens' routed experts; the weights to load are that union) and the
 * S2-MoE write-up, challenge 2 (reuse ratio |union| / (s * k), s = tokens).
 *
 *   ids         [T, k] int32 in.
 *   n_unique    [1] int32 out: U = |union|.
 *   unique      [min(E, T*k)] int32 out: the U expert ids, ascending.
 *   offsets     [min(E, T*k) + 1] int32 out: token group of unique[u] is
 *               perm positions offsets[u] .. offsets[u+1]-1; offsets[U] = T*k.
 *   perm_token  [T*k] int32 out: token of each perm position (expert
 *               ascending, then token ascending).
 *   perm_slot   [T*k] int32 out: the slot j with ids[t, j] == expert.
 *   inv         [T*k] int32 out: inv[t*k + j] = perm position of (t, j).
 *   reuse_ratio [1] fp32 out: U / (T*k) rounded once to fp32; 0 when T == 0.
 * Limits: 1 <= k <= 16, 1 <= E <= 1024, T*k <= 65536, T*E <= 1048576.
 * Device errors: MOE_DEV_BAD_ID, MOE_DEV_DUP_ID (then n_unique = 0).
 */
int moe_union_permute(const int32_t* ids, int32_t T, int32_t k, int32_t E,
                      int32_t* n_unique, int32_t* unique, int32_t* offsets,
                      int32_t* perm_token, int32_t* perm_slot, int32_t* inv,
                      float* reuse_ratio, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- expert FFN
 * One layer's expert weights.  Two layouts:
 *
 * MOE_LAYOUT_ROWMAJOR: expert-major, each expert contiguous:
 *   w_gate_up [E, 2I, H]: rows 0..I-1 are W_gate, rows I..2I-1 are W_up.
 *   w_down    [E, H, I].
 *   FP8 only: scales_gate_up [E, 2I/128, H/128] and scales_down
 *   [E, H/128, I/128] fp32; weight (r, c) of a matrix is code(r, c) *
 *   scale[r/128, c/128].  NULL for the other dtypes.
 *
 * MOE_LAYOUT_TILED (bf16 or FP8; made once at load time by moe_pack_tiled):
 * blocks of 128 bytes of the reduction dimension (C = 64 bf16 or 128 FP8
 * values), each block contiguous, so that every pipeline stage of the FFN
 * reads one 32 KB contiguous piece of HBM.
 *   w_gate_up [E][MTg][H/C][256][C], MTg = ceil(I/128): block (e, m, kb)
 *     holds rows m*128 .. m*128+127 of W_gate (columns kb*C .. kb*C+C-1)
 *     followed by the same rows of W_up; rows >= I are zero.
 *   w_down [E][MTd][I/C][128][C], MTd = ceil(H/128): block (e, m, kb)
 *     holds rows m*128 .. m*128+127 of W_down, columns kb*C .. +C-1; rows
 *     >= H are zero.
 *   FP8 block scales keep their row-major shape.
 *
 * Pointers must be 16-byte aligned.  Limits: H and I multiples of 64
 * (of 128 for FP8), E <= 1024.
 *
 * Expert residency (optional, `pool` != NULL): w_gate_up / w_down then hold
 * pool->n_slots expert slots in the layout above (slot s where expert s
 * would be) instead of all E experts, and expert e of the union is read from
 * slot pool->slot_of[e].  FP8 block scales stay indexed by expert id (all E
 * experts, resident).  See moe_stage_experts.
 */
enum { MOE_LAYOUT_ROWMAJOR = 0, MOE_LAYOUT_TILED = 1 };

/*
 * moe_expert_pool -- expert-level residency of one layer on a Grace-Blackwell
 * node: hot experts live in HBM, cold ones in the Grace (host) memory and are
 * copied over NVLink-C2C into HBM staging slots when a step's union needs
 * them.
 *
 * Defined by: S2-MoE write-up, "system implementation: expert-level
 * offloading in llama.cpp" (non-expert parameters and frequently activated
 * experts stay in device memory; any other expert is fetched on demand, from
 * host memory on a platform with separate CPU and GPU memory; the hot list
 * comes from offline profiling of activation frequencies).  The write-up
 * gives no algorithm for the fetch; this library's reading: the union of the
 * layer (known only on the device) decides, a kernel copies the cold experts
 * of the union into staging slots, in union order, without a host round trip.
 *
 *   n_slots       expert slots in the layer's device buffers (1..65536).
 *   stage_first, n_stage
 *                 slots stage_first .. stage_first+n_stage-1 are staging
 *                 slots (n_stage may be 0).  Several layers may point at the
 *                 same buffers and share one staging range: every layer's
 *                 staging starts after the previous layer's FFN finished.
 *   home_slot     device [E] int32: the slot holding resident expert e
 *                 (in [0, n_slots), outside the staging range), or -1 for
 *                 a cold expert.
 *   host_gate_up, host_down
 *                 all E experts in the layer's layout (the sizes of an
 *                 un-pooled layer), in page-locked host memory the device
 *                 can address (cudaHostAlloc / cudaHostRegister), 16-byte
 *                 aligned.  May be NULL when n_stage is 0.
 *   slot_of       device [E] int32: written by moe_stage_experts for the
 *                 experts of the union; read by the FFN for the same experts.
 */
typedef struct {
  int32_t n_slots, stage_first, n_stage;
  const int32_t* home_slot;
  const void* host_gate_up;
  const void* host_down;
  int32_t* slot_of;
} moe_expert_pool;

typedef struct {
  int32_t H, I, E, dtype, layout;
  const void* w_gate_up;
  const void* w_down;
  const float* scales_gate_up;
  const float* scales_down;
  const moe_expert_pool* pool;  /* HOST pointer, read during the call only; NULL: all E resident */
} moe_layer_weights;

/* Bytes of the tiled copies of one layer's bf16 or FP8 weights (gate/up and down,
 * written to *gate_up_bytes / *down_bytes when not NULL); returns their sum,
 * or 0 if the layer cannot be tiled. */
size_t moe_tiled_bytes(const moe_layer_weights* lw, size_t* gate_up_bytes, size_t* down_bytes);

/* Packs one layer's row-major bf16 or FP8 weights (src->layout must be ROWMAJOR, src->pool NULL)
 * into the MOE_LAYOUT_TILED layout at dst_gate_up / dst_down (caller-owned
 * device buffers of the sizes moe_tiled_bytes reports, 16-byte aligned, not
 * overlapping src).  FP8 scales are not copied: the tiled layer points at
 * the same scale tensors.  A load-time step; enqueued on `stream`. */
int moe_pack_tiled(const moe_layer_weights* src, void* dst_gate_up, void* dst_down, void* stream);

/* Bytes of one expert's gate/up and down weights in the layer's layout
 * (the size of one pool slot); returns their sum, 0 for an invalid layer. */
size_t moe_expert_bytes(const moe_layer_weights* lw, size_t* gate_up_bytes, size_t* down_bytes);

/*
 * moe_stage_experts -- makes every expert of a layer's union available in
 * the layer's device pool (lw->pool must be set).
 *
 * For u < *n_unique, expert e = unique[u]: if home_slot[e] >= 0 then
 * slot_of[e] = home_slot[e]; otherwise e is the c-th cold expert of the
 * union (c counted in union order from 0), slot_of[e] = stage_first + c, and its
 * gate/up and down weights are copied from host_gate_up / host_down into
 * that slot of w_gate_up / w_down.  The copy reads host memory with plain
 * 16-byte loads over NVLink-C2C (no bulk-tensor copies touch host memory)
 * and runs on the device: the host never sees the union.  Call it after the
 * union is written and before moe_verify_ffn on the same stream;
 * moe_verify_step does so itself for every layer that has a pool.
 *
 *   n_unique, unique   as written by moe_union_permute (device).
 *   n_staged           device int32 out, optional: cold experts copied.
 * Device errors: MOE_DEV_CAPACITY (more cold experts than staging slots:
 * the excess are not copied and their slot_of is -1, so the FFN flags them),
 * MOE_DEV_BAD_ID (an id outside [0, E), or a home slot that is neither -1
 * nor a slot outside the staging range: that expert's slot_of is -1).
 */
int moe_stage_experts(const moe_layer_weights* lw, const int32_t* n_unique, const int32_t* unique,
                      int32_t* n_staged, int32_t* dev_err, void* stream);

/*
 * moe_hot_list -- the hot-expert list of expert-level residency.
 *
 * Defined by: S2-MoE write-up, "system implementation: expert-level
 * offloading" (frequently activated experts stay resident; the list comes
 * from offline profiling of activation frequencies).  Reading: counts[e] is
 * the number of entries of ids equal to e; the hot list is the n_hot experts
 * with the largest counts, equal counts going to the lower id, written to
 * hot[] in ascending id order; home_slot[e] = first_slot + j for hot[j] and
 * -1 for every other expert (the home-slot table of moe_expert_pool, with
 * layer l's hot experts at first_slot = l * n_hot).
 *
 *   ids        [n_ids] int32 profiled routing decisions (expert ids, any
 *              layout; -1 entries are ignored).  0 <= n_ids <= 2^31 - 1.
 *   E          experts, 1..4096.   n_hot  0..E.   first_slot >= 0.
 *   counts     [E] int32 out, optional (NULL: not written).
 *   hot        [n_hot] int32 out (may be NULL when n_hot = 0).
 *   home_slot  [E] int32 out, optional.
 * One CTA; a load-time step, not on the verify path.
 * Device errors: MOE_DEV_BAD_ID (an id outside [-1, E): not counted).
 */
int moe_hot_list(const int32_t* ids, int64_t n_ids, int32_t E, int32_t n_hot, int32_t first_slot,
                 int32_t* counts, int32_t* hot, int32_t* home_slot, int32_t* dev_err, void* stream);

/* Bytes of workspace moe_verify_ffn needs for T tokens with top-k routing. */
size_t moe_verify_ffn_workspace(const moe_layer_weights* lw, int32_t T, int32_t k);

/*
 * moe_verify_ffn -- y_t = sum_{j<k} w[t,j] * FFN_{ids[t,j]}(x_t), reading the
 * weights of each expert in the union from HBM once.
 *
 * Defined by: EcoSpec write-up section 1 (an MoE layer's cost is set by the
 * union of experts the tokens activate) and the S2-MoE write-up's background
 * (each token passes its top-k experts; verification reuses loaded weights).
 * FFN_e(x) = W_down,e (silu(W_gate,e x) * (W_up,e x)), silu(a) = a/(1+e^-a).
 *
 *   x        [T, H] activations: fp32 for MOE_DTYPE_F32, bf16 bits otherwise.
 *   n_unique, unique, offsets, perm_token, inv: as written by
 *            moe_union_permute for the same ids (each expert's group lists
 *            its tokens in ascending order; with bf16 weights and T <= 32 a
 *            group that does not ascend raises MOE_DEV_BAD_ID).
 *   w        [T, k] fp32 routing weights.
 *   y        [T, H] fp32 out.  The combine sums slots j = 0..k-1 in order.
 * Arithmetic: fp32 accumulation.  bf16 weights: tensor cores on bf16
 * operands; the SwiGLU intermediate is rounded to bf16.  FP8 weights with
 * T <= 32: tensor cores on E4M3 operands, activations and the intermediate
 * carried as a per-row-scaled E4M3 pair hi + lo/16 (relative error near
 * 2^-8), block scales applied exactly in fp32 per 128-column block; larger T
 * uses CUDA cores with exact decoding.  fp32 weights: CUDA cores.
 * Limits: 1 <= T <= 256, 1 <= k <= 16.
 * Device errors: MOE_DEV_CAPACITY (n_unique > min(E, T*k)), MOE_DEV_BAD_ID.
 */
int moe_verify_ffn(const void* x, int32_t T, int32_t k, const moe_layer_weights* lw,
                   const int32_t* n_unique, const int32_t* unique, const int32_t* offsets,
                   const int32_t* perm_token, const int32_t* inv, const float* w,
                   float* y, void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * moe_verify_ffn_noalloc -- moe_verify_ffn for callers that cannot allocate
 * device memory.  The pages have no counterpart; this is a deployment aid.
 *
 * Who needs it: code running during CUDA graph capture (cudaMalloc is not
 * allowed there), plugin / custom-op hosts that own the device allocator and
 * forbid other allocations, and latency-critical serving loops where an
 * allocation would synchronise the device.  Such callers pass inputs and
 * outputs only; the scratch space lives in a static device array of 64 MiB
 * inside the library, present on every GPU that loads the library until the
 * process exits.  The call performs no cudaMalloc/cudaFree or other
 * allocating routine.
 *
 * Arguments and results: exactly those of moe_verify_ffn, without the
 * workspace.  Returns MOE_ERR_UNSUPPORTED when the FFN would need more than
 * the 64 MiB of static scratch (moe_verify_ffn_workspace() tells the size).
 * All calls on a device share the array and it keeps the previous call's
 * contents (the kernels reset what must start at zero); calls that overlap
 * on the GPU race on it.  The first call on a device looks up the array's
 * address with that device current; make it before any stream capture.
 * The address is kept per device and driver context: after a context reset
 * (cudaDeviceReset, or a framework recreating the primary context) the next
 * call looks it up again, and that call too should precede any capture.
 */
int moe_verify_ffn_noalloc(const void* x, int32_t T, int32_t k, const moe_layer_weights* lw,
                           const int32_t* n_unique, const int32_t* unique, const int32_t* offsets,
                           const int32_t* perm_token, const int32_t* inv, const float* w, float* y,
                           int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- selection
 * eco_select -- EcoSpec cost-aware draft selection, one tree per sequence.
 *
 * Defined by: EcoSpec write-up section 3.2 (expert buffer B, empty at the
 * start of every speculative step) and section 3.3 (score
 * S(t) = P(t) / (|E_traj(t) \ B| + eps); greedy: take the argmax, add it to
 * S, B |= E_traj(best), until gamma nodes are chosen; prefix consistency).
 * mode 1 is the static ablation of section 4.3: denominator |E_traj(t)|.
 * mode 2 is batch-global: one buffer B shared by all nseq sequences and one
 * greedy over the forest of their trees, with the budget
 * sum(min(gamma_i, N)) and at most min(gamma_max, N) nodes per sequence, so
 * each sequence's depth is decided by the scores (the write-up's batch
 * ablation, section 4.3, gives no algorithm; this is the plainest batch form
 * of section 3.3).  Ties go to the lower (sequence, node) index.
 *
 *   P        [nseq, N] fp32 path probabilities (product of draft
 *            probabilities from the root), finite and >= 0.
 *   parent   [nseq, N] int32: parent draft node, -1 for a child of the root;
 *            parent[t] < t (breadth-first numbering).
 *   own_fp   [nseq, N, W] uint32: each node's own predicted footprint;
 *            bit l*E + e (word (l*E+e)/32, bit (l*E+e)%32) marks (layer l,
 *            expert e).  E_traj(t) is the OR of own_fp along the path to t.
 *   gamma_per_seq [nseq] int32 per-sequence budget in [0, gamma_max], or
 *            NULL for gamma_max everywhere.  Budgets above N select all nodes.
 *   selected [nseq, gamma_max] int32 out: chosen nodes in selection order;
 *            unused slots are -1 (in mode 2 a sequence's count is whatever
 *            the greedy gave it).
 *   union_size [nseq] int32 out: |B| after the last round (mode 2: the
 *            union of that sequence's own selected trajectories).
 * Scores are compared exactly: a beats b when
 * P_a * (c_b + eps) > P_b * (c_a + eps) in exact arithmetic.  The kernel
 * writes P = m * 2^e and c + eps = X * 2^-s with X = c * 2^s + 1, and compares
 * the integer products m_a * X_b and m_b * X_a (below 2^53) scaled by the
 * exponent difference; where every X < 2^24 the correctly rounded fp32
 * quotient P / X serves as a monotone key and only key ties fall back to the
 * integer comparison.  Equal scores go to the lower node index.
 * Limits: eps = 2^-s with 0 <= s <= 20; W*32*2^s < 2^29; 1 <= N <= 1024;
 * 1 <= W <= 4096; N*W <= 40960; mode 2: nseq*N <= 1024, nseq*N*W <= 40960.
 * Device errors: MOE_DEV_BAD_TREE, MOE_DEV_BAD_PROB (that sequence's
 * selected = -1, union_size = 0).
 */
typedef struct {
  int32_t N, W, gamma_max, mode;
  float eps;
} eco_cfg;

int eco_select(const float* P, const int32_t* parent, const uint32_t* own_fp, int32_t nseq,
               const int32_t* gamma_per_seq, const eco_cfg* cfg, int32_t* selected,
               int32_t* union_size, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- whole step
 * moe_verify_step -- one verify step: selection, then for each of L layers
 * route (optionally biased) -> union/permute -> expert FFN + combine.
 *
 * Defined by: EcoSpec write-up section 2 (a round drafts a tree, selects
 * gamma nodes and verifies gamma+1 tokens in one target forward) and the
 * calls above.  Verify tokens are, per sequence, the root token followed by
 * the selected nodes in selection order; sequences are concatenated.  The
 * reuse-bias confidence of a token is its path probability (1 for a root).
 *
 *   node_logits [L, nseq, N+1, E] fp32 router logits of every tree node per
 *               layer; row 0 of each sequence is the root token.
 *   node_x      [L, nseq, N+1, H] layer inputs of every tree node (fp32 or
 *               bf16 bits, by dtype).
 *   layers      HOST array of L moe_layer_weights (same H, I, E, dtype).  A
 *               layer with an expert pool has its union's cold experts
 *               staged (moe_stage_experts) between its routing and its FFN;
 *               layers may share one staging range.
 *   selected, union_size: as eco_select.
 *   n_unique    [L] int32 out: union size per layer.
 *   y           [L, T, H] fp32 out.
 * cfg->T must equal sum over sequences of (gamma_i + 1) with gamma_i clamped
 * to N; the device checks it (MOE_DEV_CAPACITY if not).
 * Layers with tiled, resident tensor-core weights: each layer's down launch
 * also asks L2 to fetch part of the next layer's gate/up weights for the
 * experts the selection predicts (the selected nodes' footprints).  This
 * changes no result.
 */
typedef struct {
  int32_t L, nseq, N, W, E, k, H, I, dtype, layout;
  int32_t T, gamma_max, mode;
  float eps;
  int32_t use_bias, cap;
  float alpha;
} moe_step_cfg;

size_t moe_verify_step_workspace(const moe_step_cfg* cfg);

int moe_verify_step(const moe_step_cfg* cfg, const float* P, const int32_t* parent,
                    const uint32_t* own_fp, const int32_t* gamma_per_seq,
                    const float* node_logits, const void* node_x,
                    const moe_layer_weights* layers, int32_t* selected, int32_t* union_size,
                    int32_t* n_unique, float* y, void* workspace, size_t ws_bytes,
                    int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- S2-MoE expansion
 * s2_expand -- routing-aware adaptive speculative expansion: which draft
 * tokens are worth verifying, judged by the experts they would add.
 *
 * Defined by: S2-MoE write-up, component 1.  Adding draft token i to the
 * selected set S costs |E_i minus the union of E_j over j in S| * T_exp plus
 * the draft cost C_draft; its utility is p_i * T_AR over that cost; every
 * candidate with utility >= 1 is taken, until none qualifies.  Readings used:
 * on a draft tree a node is a candidate once its parent is selected (the
 * root's children always are), so the selection is prefix-closed; the
 * selected set does not depend on the order candidates are examined in (it
 * is the least fixed point of a monotone rule); U_i >= 1 is evaluated as
 * p_i * T_AR >= n_new * T_exp + C_draft in fp64 with that operation order
 * (with the cold-expert term below when cold_fp is given).
 *
 *   P          [nseq, N] fp32 path probability of each draft node (p_i).
 *   parent     [nseq, N] int32, breadth-first order: -1 or an index < t.
 *   own_fp     [nseq, N, W] uint32: node's own predicted footprint, bit
 *              l*E + e for expert e of layer l.
 *   cfg        N, W and the cost model T_AR, T_exp, C_draft, T_cold
 *              (finite, >= 0, any consistent time unit).
 *   cfg->cold_fp  optional DEVICE [W] uint32 mask of the experts that are
 *              not resident (bit l*E + e; see moe_expert_pool), or NULL.
 *              The write-up calibrates the expert cost from the expert's
 *              bytes and the bandwidth it is moved at; with expert residency
 *              a cold expert is moved twice (host link, then HBM), so each
 *              new expert that is also cold adds T_cold:
 *              cost = (n_new * T_exp + n_new_cold * T_cold) + C_draft, in
 *              fp64 in that order.  NULL (or T_cold = 0) gives the plain rule.
 *   selected   [nseq, N] int32 out: selected node indices in ascending
 *              order, then -1.
 *   n_selected [nseq] int32 out; union_size [nseq] int32 out: bits set in
 *              the union of the selected footprints.
 * Limits: 1 <= N <= 1024, 1 <= W <= 4096, N*W <= 40960.  Device errors:
 * MOE_DEV_BAD_TREE, MOE_DEV_BAD_PROB (that sequence selects nothing).
 */
typedef struct {
  int32_t N, W;
  float T_AR, T_exp, C_draft, T_cold;
  const uint32_t* cold_fp;
} s2_cfg;

int s2_expand(const float* P, const int32_t* parent, const uint32_t* own_fp, int32_t nseq,
              const s2_cfg* cfg, int32_t* selected, int32_t* n_selected, int32_t* union_size,
              int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- depth policy
 * moe_depth_policy -- the confidence-gated depth vector of ragged
 * speculation: how many draft positions each sequence of the batch should
 * verify this step.
 *
 * Defined by: the width-vs-depth note, section 2 ("where to spend depth"):
 * choose the depth vector d that maximises the expected batch throughput,
 * first one batch-common depth from the live sequences' confidences, then
 * greedy truncation of single sequences while that raises the expected
 * throughput; the draft's confidence at a depth is the cumulative product of
 * its per-token confidences.  Readings used:
 *   expected committed tokens of sequence i at depth d_i:
 *     A_i = 1 + conf[i][0] + ... + conf[i][d_i - 1];
 *   expected step cost: C0 + T_exp * U, U = the number of distinct bits in
 *     the union over the batch of fp[i][0..d_i] (position 0 = the root token,
 *     always verified), the verify-cost model of the S2-MoE write-up
 *     (component 1: T_exp per unique expert);
 *   throughput = sum_i A_i / cost;
 *   common depth: d_i = min(D', max_depth[i]) for D' = 0..D, largest
 *     throughput, equal throughputs to the smaller D';
 *   truncation: repeatedly apply the single decrement d_i -> d_i - 1 with
 *     the largest throughput if it is strictly larger than the current one
 *     (equal candidates to the lower i).
 * Arithmetic is fp64 in a fixed order with no contraction: A_i accumulates
 * in depth order from 1; the numerator sums sequences in index order from 0;
 * cost = C0 + (T_exp * U); throughput = numerator / cost.
 *
 *   conf       [nseq, D] fp32 cumulative confidences, each in [0, 1].
 *   fp         [nseq, D+1, W] uint32 predicted footprints (bit l*E + e for
 *              expert e of layer l): row 0 the root token, row j the j-th
 *              draft position.
 *   max_depth  [nseq] int32 per-sequence limits (clamped to [0, D]), or NULL.
 *   cfg        nseq in 1..256, D in 1..32, W >= 1 with
 *              nseq*(D+1)*(8 + 4*W) <= 200 KiB; C0 > 0 and T_exp >= 0,
 *              finite, any consistent time unit.
 *   depth      [nseq] int32 out: d.
 *   common_depth  [1] int32 out, optional: the batch-common depth D'.
 *   throughput [2] fp64 out, optional: at the common depth, and final.
 * One CTA; a control-path call (microseconds).  Device errors:
 * MOE_DEV_BAD_PROB (a confidence outside [0, 1] or NaN: every depth 0).
 */
typedef struct {
  int32_t nseq, D, W;
  float C0, T_exp;
} moe_depth_cfg;

int moe_depth_policy(const float* conf, const uint32_t* fp, const int32_t* max_depth,
                     const moe_depth_cfg* cfg, int32_t* depth, int32_t* common_depth,
                     double* throughput, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- plan
 * moe_verify_plan -- the control path of one verify step, without the
 * expert FFN: the selection of moe_verify_step and, for every layer, its
 * routing (with the reuse bias when cfg->use_bias) and expert union, all
 * written out.  For callers that schedule the expert FFN themselves (for
 * example, to stage the union's experts before the layer runs) and for
 * timing the control path on its own.
 *
 * Defined by: EcoSpec write-up section 2 (a round selects gamma nodes and
 * verifies gamma+1 tokens; a layer's verify experts are the union of the
 * tokens' routed experts) and sections 3.2-3.3; routing and bias as
 * moe_route, union as moe_union_permute.
 *
 *   cfg            as moe_verify_step; H, I, dtype and layout are not read.
 *   P, parent, own_fp, gamma_per_seq, node_logits   as moe_verify_step.
 *   selected       [nseq, gamma_max] int32 out, union_size [nseq] int32 out.
 *   verify_rows    [T] int32 out: node-table row of each verify token,
 *                  sequence-major, each sequence's root first.
 *   verify_conf    [T] fp32 out: path probability of each verify token
 *                  (1 for roots); the bias's confidence weights.
 *   ids, w         [L, T, k] out, as moe_route per layer.
 *   n_unique       [L]; unique [L, cap]; offsets [L, cap + 1];
 *   perm_token, perm_slot, inv [L, T*k]; reuse_ratio [L]: as
 *                  moe_union_permute per layer, with cap = min(E, T*k).
 * Needs no workspace.  Errors: as moe_verify_step's selection and routing.
 */
int moe_verify_plan(const moe_step_cfg* cfg, const float* P, const int32_t* parent,
                    const uint32_t* own_fp, const int32_t* gamma_per_seq, const float* node_logits,
                    int32_t* selected, int32_t* union_size, int32_t* verify_rows, float* verify_conf,
                    int32_t* ids, float* w, int32_t* n_unique, int32_t* unique, int32_t* offsets,
                    int32_t* perm_token, int32_t* perm_slot, int32_t* inv, float* reuse_ratio,
                    int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- timing
 * Optional per-kernel timing.  Between moe_profile_begin and moe_profile_end
 * the library records a CUDA event pair on the launching stream around each
 * of its kernel launches whose class bit is set in class_mask (at most
 * max_launches pairs; later launches are not recorded).  moe_profile_end
 * synchronises those events (host blocking) and writes, per kernel class, the
 * summed milliseconds and the launch count.  Classes: 0 eco_select, 1 route,
 * 2 union/permute, 3 FFN prep, 4 FFN gate/up, 5 FFN down, 6 combine,
 * 7 router logits, 8 S2-MoE expansion, 9 expert staging, 10 hot list,
 * 11 depth policy.
 * Not for use under stream capture.
 */
enum { MOE_PROF_CLASSES = 12 };
int moe_profile_begin(int32_t max_launches, int32_t class_mask);
int moe_profile_end(float* ms_per_class, int32_t* launches_per_class, int32_t n_classes);

/* ---------------------------------------------------------------- misc */
/* Static string for a status code. */
const char* moe_status_str(int status);

/* Number of kernels the library launched since load (host counter). */
uint64_t moe_launch_count(void);

/* Test hook, for exercising the failure paths without a fault.  The pages
 * have no counterpart.  mask is 0 (normal operation, the default) or an OR of:
 *   MOE_TEST_STALL_GATE_UP     the bf16 gate/up producer issues no copies, so
 *                              every bounded wait of that launch runs out and
 *                              the launch reports MOE_DEV_TIMEOUT;
 *   MOE_TEST_STALL_READY_FLAG  the step's layer heads do not publish the
 *                              union, so gate/up takes its slower fallback
 *                              (results unchanged).
 * Process-wide; read by the host at each launch.  Returns MOE_ERR_ARG for
 * unknown bits. */
enum { MOE_TEST_STALL_GATE_UP = 1, MOE_TEST_STALL_READY_FLAG = 2 };
int moe_test_set_stall(int32_t mask);

/* Trace ranges for a timeline tool (NVTX; the pages have no counterpart).
 * With on = 1, moe_verify_step and moe_verify_plan push a named NVTX range
 * around their enqueue ("moe_verify_step" / "moe_verify_plan"), one around
 * the selection launch ("selection") and one per layer ("layer <l>") on the
 * calling host thread; a tool such as Nsight Systems projects them onto the
 * GPU timeline of the stream.  on = 0 (the default) pushes nothing.  Host
 * only, process-wide; returns MOE_ERR_ARG for any other value.  Ranges mark
 * enqueue spans, so under stream capture they mark the capture, not the
 * graph's replays. */
int moe_set_nvtx(int32_t on);

/* Library ABI version (major * 100 + minor). */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
