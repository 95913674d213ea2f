// k_gemm_skinny.cu -- matmuls with at most 16 rows of A (one row per sequence
// while generating), on the CUDA cores.
//
// out[m, n] = sum_k A[m, k] W[n, k] (+ epilogue), m < M <= 16: the weight
// matrix W [N, K] (bf16) is the only large operand and is read exactly once,
// so the kernel is bound by HBM (or, at M = 16, by the FP32 FMA rate: 16 FMAs
// per 2-byte weight).  Layout of the work: a warp owns four weight rows and a
// share of K; its lanes stream the rows in 16-byte pieces (8 bf16, 256
// elements per warp step, fully coalesced), multiply them with the matching
// pieces of all M rows of A (read through L1: A is a few KB and shared by
// every warp), and keep 4 x 16 fp32 partial sums.  The K shares of one row
// group sit in one CTA and are added in a fixed order, so the result does not
// depend on scheduling.  Epilogues: bias, fp32 residual, GELU (the forward's
// two outputs), as in the tensor-core kernel.
#include "common.cuh"
#include "kernels.h"

#define SK_THREADS 256
#define SK_WARPS (SK_THREADS / 32)
#define SK_MB 16
#define SK_R 4  // weight rows per warp

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Sum v[0..15] over the 32 lanes of the warp; afterwards lane l holds the
// total of v[l & 15] (lanes l and l ^ 16 hold the same value).  Halving
// exchange: at each level a lane keeps one half of its values and adds the
// partner's copy of that half (16 shuffles instead of 16 x 5).
__device__ __forceinline__ float warp_reduce16(float* v, int lane) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;  // keep the upper half of the current 2*o values
#pragma unroll
    for (int i = 0; i < o; i++) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  // v[0] now holds, for value index (lane & 15), the sum over the 16 lanes
  // that share bit 4 of the lane id; add the other half of the warp
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// S: warps per row group (K shares); each CTA holds SK_WARPS / S groups of
// SK_R weight rows.
template <int S>
__global__ void __launch_bounds__(SK_THREADS)
    gemm_skinny_kernel(const GemmArgs g) {
  pdl_trigger();
  __shared__ float part[SK_WARPS][SK_R][SK_MB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = SK_WARPS / S;
  const int grp = blockIdx.x * G + warp / S, share = warp % S;
  const int n0 = grp * SK_R;
  const int M = g.M, N = g.N, K = g.K;
  const bf16* A = static_cast<const bf16*>(g.A);
  const bf16* W = static_cast<const bf16*>(g.B);
  pdl_wait();
  float acc[SK_R][SK_MB];
#pragma unroll
  for (int r = 0; r < SK_R; r++)
#pragma unroll
    for (int m = 0; m < SK_MB; m++) acc[r][m] = 0.f;
  if (n0 < N) {
    const bf16* wr[SK_R];
#pragma unroll
    for (int r = 0; r < SK_R; r++) wr[r] = W + (int64_t)min(n0 + r, N - 1) * g.ldb;  // rows past N: a copy, not stored
    for (int k = (share * 32 + lane) * 8; k < K; k += S * 256) {
      float f[SK_R][8];
#pragma unroll
      for (int r = 0; r < SK_R; r++) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wr[r] + k)), f[r]);
#pragma unroll
      for (int m = 0; m < SK_MB; m++) {
        if (m < M) {
          float a[8];
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(A + (int64_t)m * g.lda + k)), a);
#pragma unroll
          for (int r = 0; r < SK_R; r++)
#pragma unroll
            for (int i = 0; i < 8; i++) acc[r][m] = fmaf(a[i], f[r][i], acc[r][m]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < SK_R; r++) {
    const float v = warp_reduce16(acc[r], lane);
    if (lane < SK_MB) part[warp][r][lane] = v;
  }
  __syncthreads();
  // epilogue: the first warp of each group; lane = (row pair rp, m), two passes
  if (share == 0 && n0 < N) {
#pragma unroll
    for (int h = 0; h < SK_R / 2; h++) {
      const int r = 2 * h + (lane >> 4), m = lane & 15, n = n0 + r;
      if (m < M && n < N) {
        float x = 0.f;
        for (int s = 0; s < S; s++) x += part[warp + s][r][m];
        if (g.bias) x += g.bias[n];
        const int64_t o = (int64_t)m * g.ldo + n;
        if (g.epi == EPI_RESIDUAL) {
          static_cast<float*>(g.out)[o] = static_cast<const float*>(g.aux)[o] + x;
        } else if (g.epi == EPI_GELU_FWD) {
          float gl, gd;
          gelu_and_grad_hw(x, gl, gd);
          static_cast<bf16*>(g.out)[o] = __float2bfloat16_rn(gd);
          static_cast<bf16*>(g.out2)[o] = __float2bfloat16_rn(gl);
        } else if (g.out_f32) {
          static_cast<float*>(g.out)[o] = x;
        } else {
          static_cast<bf16*>(g.out)[o] = __float2bfloat16_rn(x);
        }
      }
    }
  }
}

bool gemm_skinny_applies(const GemmArgs& g) {
  return g.M >= 1 && g.M <= SK_MB && g.a_kmajor && g.b_kmajor && g.K % 8 == 0 && g.lda % 8 == 0 &&
         g.ldb % 8 == 0 && !g.colsum_out &&
         (g.epi == EPI_STORE || g.epi == EPI_RESIDUAL || g.epi == EPI_GELU_FWD);
}

void launch_gemm_skinny(LaunchCtx& c, const GemmArgs& g) {
  const int chunks = (g.K + 255) / 256;
  const int S = chunks >= 8 ? 8 : chunks >= 3 ? 4 : chunks >= 2 ? 2 : 1;
  const int G = SK_WARPS / S;
  const int groups = (g.N + SK_R - 1) / SK_R;
  const dim3 grid((groups + G - 1) / G);
  switch (S) {
    case 8: launch_pdl(c, gemm_skinny_kernel<8>, grid, dim3(SK_THREADS), 0, g); break;
    case 4: launch_pdl(c, gemm_skinny_kernel<4>, grid, dim3(SK_THREADS), 0, g); break;
    case 2: launch_pdl(c, gemm_skinny_kernel<2>, grid, dim3(SK_THREADS), 0, g); break;
    default: launch_pdl(c, gemm_skinny_kernel<1>, grid, dim3(SK_THREADS), 0, g); break;
  }
}
