// moe_verify_step: one speculative verify step, selection plus L MoE layers,
// enqueued on one stream with no host synchronisation (capturable).
//
// EcoSpec write-up, section 2: a round drafts a tree, selects gamma nodes and
// verifies gamma+1 tokens in one target forward; in every MoE layer the
// verify tokens route to their top-k experts and the union is loaded once.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "common.cuh"

namespace moe {
namespace {

// Bytes of the next layer's predicted experts' gate/up weights that a
// layer's down CTAs ask L2 to fetch once they have issued their last weight
// load (about 200 KB per CTA).  HBM is underused from the end of a down
// launch until the next layer's gate/up stream starts (the down launch's
// last CTAs, the combine, the next head); the next gate/up then reads these
// bytes from L2.  Larger budgets delay the down launch's end by more than
// they save.
constexpr long long kPrefetchBudget = 30ll << 20;

struct StepWs {
  int32_t* verify_rows;
  float* verify_conf;
  int32_t* ids;
  float* w;
  int32_t* unique;
  int32_t* offsets;
  int32_t* perm_token;
  int32_t* perm_slot;
  int32_t* inv;
  float* ratio;
  int32_t* ready;  // union-ready word of the head -> gate/up handshake
  uint32_t* pred_B;  // [nseq][W] the selection's expert buffers (predicted union)
  void* ffn;
  size_t ffn_bytes;
};

size_t step_ws(const moe_step_cfg& c, void* base, StepWs* out) {
  const size_t T = c.T, TK = static_cast<size_t>(c.T) * c.k;
  const size_t cap = static_cast<size_t>(c.E) < TK ? c.E : TK;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  size_t o_rows = take(T * 4), o_conf = take(T * 4), o_ids = take(TK * 4), o_w = take(TK * 4);
  size_t o_u = take(cap * 4), o_off = take((cap + 1) * 4), o_pt = take(TK * 4), o_ps = take(TK * 4);
  size_t o_inv = take(TK * 4), o_ratio = take(4), o_ready = take(4);
  size_t o_pred = take(static_cast<size_t>(c.nseq) * (c.W > 0 ? c.W : 0) * 4);
  moe_layer_weights lw{c.H, c.I, c.E, c.dtype, c.layout, nullptr, nullptr, nullptr, nullptr};
  size_t fb = ffn_workspace_bytes(lw, c.T, c.k);
  size_t o_ffn = take(fb);
  if (out) {
    char* b = static_cast<char*>(base);
    out->verify_rows = reinterpret_cast<int32_t*>(b + o_rows);
    out->verify_conf = reinterpret_cast<float*>(b + o_conf);
    out->ids = reinterpret_cast<int32_t*>(b + o_ids);
    out->w = reinterpret_cast<float*>(b + o_w);
    out->unique = reinterpret_cast<int32_t*>(b + o_u);
    out->offsets = reinterpret_cast<int32_t*>(b + o_off);
    out->perm_token = reinterpret_cast<int32_t*>(b + o_pt);
    out->perm_slot = reinterpret_cast<int32_t*>(b + o_ps);
    out->inv = reinterpret_cast<int32_t*>(b + o_inv);
    out->ratio = reinterpret_cast<float*>(b + o_ratio);
    out->ready = reinterpret_cast<int32_t*>(b + o_ready);
    out->pred_B = reinterpret_cast<uint32_t*>(b + o_pred);
    out->ffn = b + o_ffn;
    out->ffn_bytes = fb;
  }
  return off;
}

// Selection and routing limits (the control path of the step).
int plan_validate(const moe_step_cfg& c) {
  if (c.L < 1 || c.nseq < 1 || c.T < 1) return MOE_ERR_ARG;
  if (c.T < c.nseq) return MOE_ERR_ARG;
  eco_cfg ec{c.N, c.W, c.gamma_max, c.mode, c.eps};
  int st = eco_validate(ec, c.nseq);
  if (st != MOE_OK) return st;
  if (static_cast<long long>(c.L) * c.E > static_cast<long long>(c.W) * 32) return MOE_ERR_ARG;
  moe_route_cfg rc{c.T, c.E, c.k, c.use_bias, c.cap, c.alpha};
  if ((st = route_validate(rc, true)) != MOE_OK) return st;
  return union_validate(c.T, c.k, c.E);
}

int step_validate(const moe_step_cfg& c) {
  if (c.L < 1 || c.nseq < 1 || c.T < 1) return MOE_ERR_ARG;
  if (c.T < c.nseq) return MOE_ERR_ARG;
  eco_cfg ec{c.N, c.W, c.gamma_max, c.mode, c.eps};
  int st = eco_validate(ec, c.nseq);
  if (st != MOE_OK) return st;
  if (static_cast<long long>(c.L) * c.E > static_cast<long long>(c.W) * 32) return MOE_ERR_ARG;
  moe_route_cfg rc{c.T, c.E, c.k, c.use_bias, c.cap, c.alpha};
  if ((st = route_validate(rc, true)) != MOE_OK) return st;
  if ((st = union_validate(c.T, c.k, c.E)) != MOE_OK) return st;
  moe_layer_weights lw{c.H, c.I, c.E, c.dtype, c.layout, reinterpret_cast<void*>(256),
                       reinterpret_cast<void*>(256), reinterpret_cast<float*>(256),
                       reinterpret_cast<float*>(256)};
  return ffn_validate(lw, c.T, c.k);
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_verify_step_workspace(const moe_step_cfg* cfg) {
  if (!cfg || moe::step_validate(*cfg) != MOE_OK) return 0;
  return moe::step_ws(*cfg, nullptr, nullptr);
}

extern "C" int moe_verify_step(const moe_step_cfg* cfg, const float* P, const int32_t* parent,
                               const uint32_t* own_fp, const int32_t* gamma_per_seq,
                               const float* node_logits, const void* node_x,
                               const moe_layer_weights* layers, int32_t* selected,
                               int32_t* union_size, int32_t* n_unique, float* y, void* workspace,
                               size_t ws_bytes, int32_t* dev_err, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_ARG;
  const moe_step_cfg& c = *cfg;
  int st = step_validate(c);
  if (st != MOE_OK) return st;
  if (!P || !parent || !own_fp || !node_logits || !node_x || !layers || !union_size || !n_unique ||
      !y || (c.gamma_max > 0 && !selected))
    return MOE_ERR_ARG;
  if (!workspace || ws_bytes < step_ws(c, nullptr, nullptr)) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MOE_ERR_ARG;
  for (int l = 0; l < c.L; ++l) {
    const moe_layer_weights& lw = layers[l];
    if (lw.H != c.H || lw.I != c.I || lw.E != c.E || lw.dtype != c.dtype || lw.layout != c.layout)
      return MOE_ERR_ARG;
    if ((st = ffn_validate(lw, c.T, c.k)) != MOE_OK) return st;
    if (lw.pool && (st = stage_validate(lw)) != MOE_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepWs ws;
  step_ws(c, workspace, &ws);
  NvtxRange trace_step("moe_verify_step");

  EcoArgs ea{P, parent, own_fp, c.nseq, gamma_per_seq, {c.N, c.W, c.gamma_max, c.mode, c.eps},
             selected, union_size, dev_err, ws.verify_rows, ws.verify_conf, c.T, s, ws.ready, ws.pred_B};
  {
    NvtxRange trace_sel("selection");
    if ((st = eco_launch(ea)) != MOE_OK) return st;
  }

  // Test hook for the handshake's fallback (no fault is involved): after
  // moe_test_set_stall(MOE_TEST_STALL_READY_FLAG) the heads never publish the
  // union, so every gate/up launch waits out its bounded handshake and reads
  // the union after its dependency wait instead; results are unchanged.
  const bool stall_ready = (test_stall_mask() & MOE_TEST_STALL_READY_FLAG) != 0;
  const int rows = c.nseq * (c.N + 1);
  const size_t xelem = c.dtype == MOE_DTYPE_F32 ? 4 : 2;
  char layer_name[24];
  for (int l = 0; l < c.L; ++l) {
    snprintf(layer_name, sizeof(layer_name), "layer %d", l);
    NvtxRange trace_layer(layer_name);
    RouteArgs ra{node_logits + static_cast<size_t>(l) * rows * c.E, ws.verify_rows, rows,
                 c.use_bias ? ws.verify_conf : nullptr, {c.T, c.E, c.k, c.use_bias, c.cap, c.alpha},
                 ws.ids, ws.w, dev_err, s};
    const char* xl = static_cast<const char*>(node_x) + static_cast<size_t>(l) * rows * c.H * xelem;
    // bf16 tensor-core layers with T <= 32 and resident weights: the head
    // also does the FFN's prep work and hands the union to gate/up directly.
    HeadPrep hp{};
    const bool head_prep = ffn_head_prep(layers[l], c.T, c.k, ws.ffn, &hp);
    if (head_prep) {
      hp.x = reinterpret_cast<const uint16_t*>(xl);
      hp.x_rows = ws.verify_rows;
      hp.x_rows_limit = rows;
      hp.ready_flag = stall_ready ? nullptr : ws.ready;
      hp.ready_value = l % 65535 + 1;  // nonzero, 16 bits, differs from the previous layer's
    }
    // The verify rows come from the selection kernel, which the first layer's
    // head follows directly; later heads may read them before their wait.
    if ((st = layer_head_launch(ra, n_unique + l, ws.unique, ws.offsets, ws.perm_token, ws.perm_slot, ws.inv,
                                ws.ratio, true, l > 0, head_prep ? &hp : nullptr)) != MOE_OK)
      return st;
    // Expert residency: the union's cold experts are staged into HBM before
    // the FFN's prep kernel, whose wait then covers the copies (the FFN's
    // weight loads may start right after prep's wait).
    if (layers[l].pool &&
        (st = stage_launch(layers[l], n_unique + l, ws.unique, nullptr, dev_err, s, true)) != MOE_OK)
      return st;
    FfnArgs fa{xl, ws.verify_rows, rows, c.T, c.k, layers[l], n_unique + l, ws.unique, ws.offsets,
               ws.perm_token, ws.inv, ws.w, y + static_cast<size_t>(l) * c.T * c.H, ws.ffn,
               ws.ffn_bytes, dev_err, s, true, head_prep, ws.ready, l % 65535 + 1};
    // The next layer's predicted experts (the selection's buffers B), for
    // the L2 prefetch at the end of this layer's down launch.
    if (l + 1 < c.L && c.W > 0) {
      const moe_layer_weights& nx = layers[l + 1];
      const int eb = nx.dtype == MOE_DTYPE_BF16 ? 2 : (nx.dtype == MOE_DTYPE_E4M3_B128 ? 1 : 0);
      if (eb && nx.layout == MOE_LAYOUT_TILED && !nx.pool) {
        fa.pf.base = static_cast<const uint8_t*>(nx.w_gate_up);
        fa.pf.expert_bytes = static_cast<long long>((nx.I + 127) / 128) * 256 * nx.H * eb;
        fa.pf.budget = kPrefetchBudget;
        fa.pf.pred_B = ws.pred_B;
        fa.pf.rows = c.nseq;
        fa.pf.W = c.W;
        fa.pf.bit0 = (l + 1) * c.E;
      }
    }
    if ((st = ffn_launch(fa)) != MOE_OK) return st;
  }
  return MOE_OK;
}

extern "C" int moe_verify_plan(const moe_step_cfg* cfg, const float* P, const int32_t* parent,
                               const uint32_t* own_fp, const int32_t* gamma_per_seq, const float* node_logits,
                               int32_t* selected, int32_t* union_size, int32_t* verify_rows,
                               float* verify_conf, int32_t* ids, float* w, int32_t* n_unique, int32_t* unique,
                               int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, int32_t* inv,
                               float* reuse_ratio, int32_t* dev_err, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_ARG;
  const moe_step_cfg& c = *cfg;
  int st = plan_validate(c);
  if (st != MOE_OK) return st;
  if (!P || !parent || !own_fp || !node_logits || !union_size || !verify_rows || !verify_conf || !ids || !w ||
      !n_unique || !unique || !offsets || !perm_token || !perm_slot || !inv || !reuse_ratio ||
      (c.gamma_max > 0 && !selected))
    return MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  NvtxRange trace_plan("moe_verify_plan");
  EcoArgs ea{P, parent, own_fp, c.nseq, gamma_per_seq, {c.N, c.W, c.gamma_max, c.mode, c.eps},
             selected, union_size, dev_err, verify_rows, verify_conf, c.T, s};
  {
    NvtxRange trace_sel("selection");
    if ((st = eco_launch(ea)) != MOE_OK) return st;
  }
  const int rows = c.nseq * (c.N + 1);
  const size_t TK = static_cast<size_t>(c.T) * c.k;
  const size_t cap = static_cast<size_t>(c.E) < TK ? c.E : TK;
  char layer_name[24];
  for (int l = 0; l < c.L; ++l) {
    snprintf(layer_name, sizeof(layer_name), "layer %d", l);
    NvtxRange trace_layer(layer_name);
    RouteArgs ra{node_logits + static_cast<size_t>(l) * rows * c.E, verify_rows, rows,
                 c.use_bias ? verify_conf : nullptr, {c.T, c.E, c.k, c.use_bias, c.cap, c.alpha},
                 ids + l * TK, w + l * TK, dev_err, s};
    if ((st = layer_head_launch(ra, n_unique + l, unique + l * cap, offsets + l * (cap + 1), perm_token + l * TK,
                                perm_slot + l * TK, inv + l * TK, reuse_ratio + l, true, l > 0)) != MOE_OK)
      return st;
  }
  return check_launch();
}
