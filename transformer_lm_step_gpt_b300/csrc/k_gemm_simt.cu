// k_gemm_simt.cu -- the fp32-exact matmul (GPT2_FP32 mode).
//
// out[m, n] = sum_k A(m,k) B(n,k) with every product an fp32 FFMA (no TF32,
// no bf16) and the GeekNews "Linear" epilogue (bias added over rows) plus
// the fused GELU / residual / GELU-backward / accumulate variants the step
// needs.  64x64 output tile per 256-thread block, 4x4 per thread, K staged
// through shared memory 16 at a time.  Either operand may be K-major or
// M/N-major, which covers the forward (x W^T), the data gradient (dy W) and
// the weight gradient (dy^T x) without transposed copies.
#include "common.cuh"
#include "kernels.h"

#define SG_BM 64
#define SG_BN 64
#define SG_BK 16

__device__ __forceinline__ float epi_apply(const GemmArgs& g, int m, int n, float acc) {
  if (g.bias) acc += g.bias[n];
  return acc;
}

__global__ void __launch_bounds__(256) gemm_f32_kernel(GemmArgs g) {
  pdl_trigger();
  pdl_wait();
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  const float* A = static_cast<const float*>(g.A);
  const float* B = static_cast<const float*>(g.B);
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += SG_BK) {
#pragma unroll
    for (int r = 0; r < 4; r++) {
      const int idx = tid + 256 * r;
      int mm, kk;
      if (g.a_kmajor) { mm = idx / SG_BK; kk = idx % SG_BK; }
      else { kk = idx / SG_BM; mm = idx % SG_BM; }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < g.M && gk < g.K) v = g.a_kmajor ? A[(int64_t)gm * g.lda + gk] : A[(int64_t)gk * g.lda + gm];
      As[kk][mm] = v;
      int nn;
      if (g.b_kmajor) { nn = idx / SG_BK; kk = idx % SG_BK; }
      else { kk = idx / SG_BN; nn = idx % SG_BN; }
      const int gn = n0 + nn;
      const int gk2 = k0 + kk;
      float w = 0.f;
      if (gn < g.N && gk2 < g.K) w = g.b_kmajor ? B[(int64_t)gn * g.ldb + gk2] : B[(int64_t)gk2 * g.ldb + gn];
      Bs[kk][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; kk++) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; i++) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; j++) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int64_t orow = g.out_row ? (int64_t)(*g.out_row) * g.out_row_stride : 0;
  float* out = static_cast<float*>(g.out) + orow;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      const int64_t o = (int64_t)m * g.ldo + n;
      float v = acc[i][j];
      switch (g.epi) {
        case EPI_STORE: out[o] = epi_apply(g, m, n, v); break;
        case EPI_GELU_FWD: {
          v = epi_apply(g, m, n, v);
          out[o] = gelu_grad_f(v);
          static_cast<float*>(g.out2)[orow + o] = gelu_f(v);
        } break;
        case EPI_RESIDUAL: out[o] = static_cast<const float*>(g.aux)[o] + epi_apply(g, m, n, v); break;
        case EPI_MUL_AUX: out[o] = v * static_cast<const float*>(g.aux)[o]; break;
        case EPI_ACCUM: out[o] += v; break;
      }
    }
  }
}

void launch_gemm_f32(LaunchCtx& c, const GemmArgs& g) {
  dim3 grid((g.N + SG_BN - 1) / SG_BN, (g.M + SG_BM - 1) / SG_BM);
  launch_pdl(c, gemm_f32_kernel, dim3(grid), dim3(256), 0, g);
}
