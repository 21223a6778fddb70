// Internal interface between the FFN front end and its kernel paths.
#pragma once

#include "common.cuh"

namespace moe {

// Carve-up of the caller's FFN workspace.
struct FfnWorkspace {
  void* h;        // SwiGLU intermediate, [T*k, I] (fp32 for the fp32 dtype, bf16 otherwise)
  float* o;       // per-(token, slot) expert outputs, [T*k, H] fp32
};

FfnWorkspace ffn_carve(const moe_layer_weights& lw, int T, int k, void* base);
int ffn_simt_launch(const FfnArgs& a, const FfnWorkspace& ws);
int combine_launch(const FfnArgs& a, const float* o, bool pdl);

// Tensor-core path (bf16 weights).
bool ffn_tc_supported(const moe_layer_weights& lw, int T, int k);
size_t ffn_tc_workspace_bytes(const moe_layer_weights& lw, int T, int k);
int ffn_tc_launch(const FfnArgs& a);
bool ffn_tc_head_prep(const moe_layer_weights& lw, int T, int k, void* ws, HeadPrep* hp);

// Tensor-core path (FP8 E4M3 weights with 128 x 128 block scales).
bool ffn_fp8_supported(const moe_layer_weights& lw, int T, int k);
size_t ffn_fp8_workspace_bytes(const moe_layer_weights& lw, int T, int k);
int ffn_fp8_launch(const FfnArgs& a);
bool ffn_fp8_head_prep(const moe_layer_weights& lw, int T, int k, void* ws, HeadPrep* hp);

}  // namespace moe
