// k_attn_tc.cu -- bf16 causal attention entry points.
// Bring-up version: routes to the CUDA-core kernels of k_attn_simt.cu.
#include "common.cuh"
#include "kernels.h"

void launch_attention_fwd_bf16(LaunchCtx& c, bf16* y, float* lse, const bf16* qkv, int B, int T,
                               int C, int NH) {
  launch_attention_fwd_simt<bf16>(c, y, lse, qkv, B, T, C, NH);
}

void launch_attention_bwd_bf16(LaunchCtx& c, bf16* dqkv, const bf16* dy, const bf16* y,
                               const bf16* qkv, const float* lse, float* dsum, int B, int T,
                               int C, int NH) {
  launch_attention_bwd_simt<bf16>(c, dqkv, dy, y, qkv, lse, dsum, B, T, C, NH, nullptr);
}
