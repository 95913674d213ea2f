// k_attn_simt.cu -- causal multi-head self-attention on CUDA cores.
//
// GeekNews, "A GPT-2-based ChatGPT clone in 3000 bytes of C", section "The
// Transformer core": q, k, v from one Linear, split per head, q k^T, the
// lower-triangular causal mask, softmax, times v, heads merged.  Scale
// 1/sqrt(hs).  This is the fp32-exact path: one warp per query row (forward,
// dq) or key row (dk, dv), scores staged in shared memory, fp32 arithmetic
// throughout.  The backward recomputes the probabilities from the saved
// row logsumexp and never materialises T x T.  It is deterministic: dq and
// (dk, dv) are produced by separate kernels, each summing in index order.
#include "common.cuh"
#include "kernels.h"

#define AS_WARPS 4

template <typename T>
__global__ void attn_fwd_simt_kernel(T* y, float* lse, const T* qkv, int Tn, int C, int NH) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sc[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * AS_WARPS + warp, h = blockIdx.y, b = blockIdx.z;
  if (t >= Tn) return;
  const int hs = C / NH;
  const int64_t C3 = 3 * (int64_t)C;
  const float scale = 1.f / sqrtf((float)hs);
  const T* q = qkv + ((int64_t)b * Tn + t) * C3 + h * hs;
  float* s = sc + warp * Tn;
  float mx = -INFINITY;
  for (int j = lane; j <= t; j += 32) {
    const T* k = qkv + ((int64_t)b * Tn + j) * C3 + C + h * hs;
    float d = 0.f;
    for (int i = 0; i < hs; i++) d += to_f(q[i]) * to_f(k[i]);
    d = d * scale;
    s[j] = d;
    mx = fmaxf(mx, d);
  }
  mx = warp_max(mx);
  float sum = 0.f;
  for (int j = lane; j <= t; j += 32) {
    const float e = expf(s[j] - mx);
    s[j] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  __syncwarp();
  for (int i = lane; i < hs; i += 32) {
    float acc = 0.f;
    for (int j = 0; j <= t; j++) acc += (s[j] / sum) * to_f(qkv[((int64_t)b * Tn + j) * C3 + 2 * C + h * hs + i]);
    y[((int64_t)b * Tn + t) * C + h * hs + i] = from_f<T>(acc);
  }
  if (lane == 0) lse[((int64_t)b * NH + h) * Tn + t] = mx + logf(sum);
}

// dq for query row t, and D_t = sum_i dy_i y_i saved for the dk/dv kernel:
//   p_j = exp(s_j - lse_t), dp_j = dy . v_j, ds_j = p_j (dp_j - D_t),
//   dq = scale * sum_j ds_j k_j.
template <typename T>
__global__ void attn_bwd_dq_simt_kernel(T* dqkv, float* dsum, const T* dy, const T* y,
                                        const T* qkv, const float* lse, int Tn, int C, int NH) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sc[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * AS_WARPS + warp, h = blockIdx.y, b = blockIdx.z;
  if (t >= Tn) return;
  const int hs = C / NH;
  const int64_t C3 = 3 * (int64_t)C;
  const float scale = 1.f / sqrtf((float)hs);
  const T* dyr = dy + ((int64_t)b * Tn + t) * C + h * hs;
  const T* yr = y + ((int64_t)b * Tn + t) * C + h * hs;
  float D = 0.f;
  for (int i = lane; i < hs; i += 32) D += to_f(dyr[i]) * to_f(yr[i]);
  D = warp_sum(D);
  const int64_t bh = (int64_t)b * NH + h;
  if (lane == 0) dsum[bh * Tn + t] = D;
  const float L = lse[bh * Tn + t];
  const T* q = qkv + ((int64_t)b * Tn + t) * C3 + h * hs;
  float* ds = sc + warp * Tn;
  for (int j = lane; j <= t; j += 32) {
    const T* k = qkv + ((int64_t)b * Tn + j) * C3 + C + h * hs;
    const T* v = k + C;
    float s = 0.f, dp = 0.f;
    for (int i = 0; i < hs; i++) { s += to_f(q[i]) * to_f(k[i]); dp += to_f(dyr[i]) * to_f(v[i]); }
    const float p = expf(s * scale - L);
    ds[j] = p * (dp - D);
  }
  __syncwarp();
  for (int i = lane; i < hs; i += 32) {
    float acc = 0.f;
    for (int j = 0; j <= t; j++) acc += ds[j] * to_f(qkv[((int64_t)b * Tn + j) * C3 + C + h * hs + i]);
    dqkv[((int64_t)b * Tn + t) * C3 + h * hs + i] = from_f<T>(acc * scale);
  }
}

// dk, dv for key row j: over queries t >= j,
//   dv = sum_t p_tj dy_t,  dk = scale * sum_t ds_tj q_t.
template <typename T>
__global__ void attn_bwd_dkv_simt_kernel(T* dqkv, const float* dsum, const T* dy, const T* qkv,
                                         const float* lse, int Tn, int C, int NH) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sc[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * AS_WARPS + warp, h = blockIdx.y, b = blockIdx.z;
  if (j >= Tn) return;
  const int hs = C / NH;
  const int64_t C3 = 3 * (int64_t)C;
  const float scale = 1.f / sqrtf((float)hs);
  const int64_t bh = (int64_t)b * NH + h;
  const T* k = qkv + ((int64_t)b * Tn + j) * C3 + C + h * hs;
  const T* v = k + C;
  float* P = sc + warp * 2 * Tn;
  float* DS = P + Tn;
  for (int t = j + lane; t < Tn; t += 32) {
    const T* q = qkv + ((int64_t)b * Tn + t) * C3 + h * hs;
    const T* dyr = dy + ((int64_t)b * Tn + t) * C + h * hs;
    float s = 0.f, dp = 0.f;
    for (int i = 0; i < hs; i++) { s += to_f(q[i]) * to_f(k[i]); dp += to_f(dyr[i]) * to_f(v[i]); }
    const float p = expf(s * scale - lse[bh * Tn + t]);
    P[t] = p;
    DS[t] = p * (dp - dsum[bh * Tn + t]);
  }
  __syncwarp();
  for (int i = lane; i < hs; i += 32) {
    float ak = 0.f, av = 0.f;
    for (int t = j; t < Tn; t++) {
      ak += DS[t] * to_f(qkv[((int64_t)b * Tn + t) * C3 + h * hs + i]);
      av += P[t] * to_f(dy[((int64_t)b * Tn + t) * C + h * hs + i]);
    }
    dqkv[((int64_t)b * Tn + j) * C3 + C + h * hs + i] = from_f<T>(ak * scale);
    dqkv[((int64_t)b * Tn + j) * C3 + 2 * C + h * hs + i] = from_f<T>(av);
  }
}

template <typename T>
void launch_attention_fwd_simt(LaunchCtx& c, T* y, float* lse, const T* qkv, int B, int Tn, int C,
                               int NH) {
  dim3 grid((Tn + AS_WARPS - 1) / AS_WARPS, NH, B);
  const size_t smem = (size_t)AS_WARPS * Tn * sizeof(float);
  cudaFuncSetAttribute(attn_fwd_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(c, attn_fwd_simt_kernel<T>, dim3(grid), dim3(AS_WARPS * 32), smem, y, lse, qkv, Tn, C, NH);
}

int64_t attention_simt_scratch_floats(int B, int Tn, int NH) { return (int64_t)B * NH * Tn; }

template <typename T>
void launch_attention_bwd_simt(LaunchCtx& c, T* dqkv, const T* dy, const T* y, const T* qkv,
                               const float* lse, float* dsum, int B, int Tn, int C, int NH,
                               float* scratch) {
  (void)scratch;
  dim3 grid((Tn + AS_WARPS - 1) / AS_WARPS, NH, B);
  size_t smem = (size_t)AS_WARPS * Tn * sizeof(float);
  cudaFuncSetAttribute(attn_bwd_dq_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(c, attn_bwd_dq_simt_kernel<T>, dim3(grid), dim3(AS_WARPS * 32), smem, dqkv, dsum, dy, y, qkv, lse, Tn, C, NH);
  smem = (size_t)AS_WARPS * 2 * Tn * sizeof(float);
  cudaFuncSetAttribute(attn_bwd_dkv_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(c, attn_bwd_dkv_simt_kernel<T>, dim3(grid), dim3(AS_WARPS * 32), smem, dqkv, dsum, dy, qkv, lse, Tn, C, NH);
}

template void launch_attention_fwd_simt<float>(LaunchCtx&, float*, float*, const float*, int, int, int, int);
template void launch_attention_fwd_simt<bf16>(LaunchCtx&, bf16*, float*, const bf16*, int, int, int, int);
template void launch_attention_bwd_simt<float>(LaunchCtx&, float*, const float*, const float*, const float*,
                                               const float*, float*, int, int, int, int, float*);
template void launch_attention_bwd_simt<bf16>(LaunchCtx&, bf16*, const bf16*, const bf16*, const bf16*,
                                              const float*, float*, int, int, int, int, float*);
