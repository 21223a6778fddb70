// moe_verify_ffn front end: argument checks, workspace layout and the choice
// of kernel path.
#include "common.cuh"
#include "ffn_internal.cuh"

namespace moe {

namespace {
size_t elem_bytes_h(const moe_layer_weights& lw) { return lw.dtype == MOE_DTYPE_F32 ? 4 : 2; }
}  // namespace

size_t ffn_simt_workspace_bytes(const moe_layer_weights& lw, int T, int k) {
  const size_t TK = static_cast<size_t>(T) * k;
  size_t b = 0;
  b += align_up(TK * lw.I * elem_bytes_h(lw), 256);
  b += align_up(TK * lw.H * sizeof(float), 256);
  return b;
}

size_t ffn_workspace_bytes(const moe_layer_weights& lw, int T, int k) {
  if (ffn_tc_supported(lw, T, k)) return ffn_tc_workspace_bytes(lw, T, k);
  if (ffn_fp8_supported(lw, T, k)) return ffn_fp8_workspace_bytes(lw, T, k);
  return ffn_simt_workspace_bytes(lw, T, k);
}

FfnWorkspace ffn_carve(const moe_layer_weights& lw, int T, int k, void* base) {
  const size_t TK = static_cast<size_t>(T) * k;
  char* p = static_cast<char*>(base);
  FfnWorkspace ws;
  ws.h = p;
  p += align_up(TK * lw.I * elem_bytes_h(lw), 256);
  ws.o = reinterpret_cast<float*>(p);
  return ws;
}

int ffn_validate(const moe_layer_weights& lw, int T, int k) {
  if (lw.dtype != MOE_DTYPE_F32 && lw.dtype != MOE_DTYPE_BF16 && lw.dtype != MOE_DTYPE_E4M3_B128)
    return MOE_ERR_UNSUPPORTED;
  if (T < 0 || T > 256 || k < 1 || k > 16) return MOE_ERR_UNSUPPORTED;
  if (lw.E < 1 || lw.E > 1024 || lw.H < 64 || lw.I < 64) return MOE_ERR_UNSUPPORTED;
  const int mult = lw.dtype == MOE_DTYPE_E4M3_B128 ? 128 : 64;
  if (lw.H % mult || lw.I % mult) return MOE_ERR_UNSUPPORTED;
  if (lw.layout != MOE_LAYOUT_ROWMAJOR && lw.layout != MOE_LAYOUT_TILED) return MOE_ERR_ARG;
  if (lw.layout == MOE_LAYOUT_TILED && lw.dtype == MOE_DTYPE_F32) return MOE_ERR_UNSUPPORTED;
  if (!lw.w_gate_up || !lw.w_down) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(lw.w_gate_up) | reinterpret_cast<uintptr_t>(lw.w_down)) & 15)
    return MOE_ERR_ARG;
  if (lw.dtype == MOE_DTYPE_E4M3_B128 && (!lw.scales_gate_up || !lw.scales_down)) return MOE_ERR_ARG;
  if (lw.pool) {
    const moe_expert_pool& pl = *lw.pool;
    if (pl.n_slots < 1 || pl.n_slots > 65536 || pl.stage_first < 0 || pl.n_stage < 0 ||
        pl.stage_first > pl.n_slots - pl.n_stage || !pl.slot_of)
      return MOE_ERR_ARG;
    // Tile-block indices of the slots must stay within int range.
    const long long blocks_gu = static_cast<long long>((lw.I + 127) / 128) * (lw.H / 64);
    const long long blocks_d = static_cast<long long>((lw.H + 127) / 128) * (lw.I / 64);
    const long long mb = blocks_gu > blocks_d ? blocks_gu : blocks_d;
    if (pl.n_slots * mb >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

bool ffn_head_prep(const moe_layer_weights& lw, int T, int k, void* ws, HeadPrep* hp) {
  if (ffn_tc_supported(lw, T, k)) return ffn_tc_head_prep(lw, T, k, ws, hp);
  if (ffn_fp8_supported(lw, T, k)) return ffn_fp8_head_prep(lw, T, k, ws, hp);
  return false;
}

int ffn_launch(const FfnArgs& a) {
  if (a.T == 0) return MOE_OK;
  if (a.ws_bytes < ffn_workspace_bytes(a.lw, a.T, a.k) || !a.ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(a.ws) & 255) return MOE_ERR_ARG;
  if (ffn_tc_supported(a.lw, a.T, a.k)) return ffn_tc_launch(a);
  if (ffn_fp8_supported(a.lw, a.T, a.k)) return ffn_fp8_launch(a);
  if (a.lw.layout != MOE_LAYOUT_ROWMAJOR) return MOE_ERR_UNSUPPORTED;  // CUDA-core path reads row-major only
  FfnWorkspace ws = ffn_carve(a.lw, a.T, a.k, a.ws);
  return ffn_simt_launch(a, ws);
}

}  // namespace moe

extern "C" size_t moe_verify_ffn_workspace(const moe_layer_weights* lw, int32_t T, int32_t k) {
  if (!lw || moe::ffn_validate(*lw, T, k) != MOE_OK) return 0;
  return moe::ffn_workspace_bytes(*lw, T, k);
}

extern "C" int moe_verify_ffn(const void* x, int32_t T, int32_t k, const moe_layer_weights* lw,
                              const int32_t* n_unique, const int32_t* unique, const int32_t* offsets,
                              const int32_t* perm_token, const int32_t* inv, const float* w,
                              float* y, void* workspace, size_t ws_bytes, int32_t* dev_err,
                              void* stream) {
  if (!lw) return MOE_ERR_ARG;
  int st = moe::ffn_validate(*lw, T, k);
  if (st != MOE_OK) return st;
  if (T > 0 && (!x || !n_unique || !unique || !offsets || !perm_token || !inv || !w || !y))
    return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return MOE_ERR_ARG;
  moe::FfnArgs a{x, nullptr, 0, T, k, *lw, n_unique, unique, offsets, perm_token, inv, w, y,
                 workspace, ws_bytes, dev_err, static_cast<cudaStream_t>(stream)};
  return moe::ffn_launch(a);
}
