// Times the library's bf16 matmul (launch_gemm_bf16: the CTA-pair tcgen05
// kernel at these sizes) on the fifteen products of one GPT-2 124M training
// step at B=16, T=1024 (the four Linear layers' forward, data-gradient and
// weight-gradient products and the tied head's), with the epilogue each one
// has in the step.  Each shape runs 5 warm-up and 20 timed launches back to
// back (CUDA events) after a 0.5 s rest, so that the clock recovers between
// shapes.  Prints one JSON object: per shape the microseconds per launch and
// TFLOP/s, and the device error word.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <unistd.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>
#include "kernels.h"

__global__ void fill_bf16(__nv_bfloat16* p, size_t n, unsigned seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    unsigned h = (unsigned)i * 2654435761u ^ seed;
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    h ^= h >> 15;
    p[i] = __float2bfloat16(((h & 0xffff) / 65536.f - 0.5f) * 0.1f);
  }
}
__global__ void fill_f32(float* p, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = 0.01f * (float)(i % 7);
}

int main() {
  const int B = 16, T = 1024, C = 768, Vp = 50304, M = B * T;
  if (!gemm_bf16_init()) { printf("{\"error\": \"no tensor-map encoder\"}\n"); return 1; }
  auto alloc = [](size_t n) {
    void* p = nullptr;
    if (cudaMalloc(&p, n) != cudaSuccess) { printf("{\"error\": \"cudaMalloc\"}\n"); exit(1); }
    return p;
  };
  // the largest operand of each role: A up to M x Vp (dlogits), W up to
  // max(Vp x C, M x 4C) elements (an N-major operand with K = M rows)
  const size_t nA = (size_t)M * Vp, nW = std::max((size_t)Vp * C, (size_t)M * 4 * C);
  __nv_bfloat16* A = (__nv_bfloat16*)alloc(nA * 2);
  __nv_bfloat16* W = (__nv_bfloat16*)alloc(nW * 2);
  __nv_bfloat16* O = (__nv_bfloat16*)alloc(nA * 2);
  __nv_bfloat16* O2 = (__nv_bfloat16*)alloc((size_t)M * 4 * C * 2);
  __nv_bfloat16* AUXB = (__nv_bfloat16*)alloc((size_t)M * 4 * C * 2);
  float* OF = (float*)alloc((size_t)M * C * 4);
  float* AUXF = (float*)alloc((size_t)M * C * 4);
  float* G = (float*)alloc((size_t)Vp * C * 4);
  float* bias = (float*)alloc(4 * 65536);
  float* splitk = (float*)alloc(sizeof(float) * 16 * C * C);
  int* flags = (int*)alloc(sizeof(int) * 8192);
  float* colsum = (float*)alloc(sizeof(float) * (M / 32) * 4 * C);
  float* dsum = (float*)alloc(sizeof(float) * M * 12);
  int* err = (int*)alloc(4);
  cudaMemset(flags, 0, sizeof(int) * 8192);
  cudaMemset(err, 0, 4);
  fill_bf16<<<1184, 256>>>(A, nA, 1);
  fill_bf16<<<1184, 256>>>(W, nW, 2);
  fill_bf16<<<1184, 256>>>(AUXB, (size_t)M * 4 * C, 3);
  fill_f32<<<1184, 256>>>(AUXF, (size_t)M * C);
  fill_f32<<<1184, 256>>>(G, (size_t)Vp * C);
  fill_f32<<<64, 256>>>(bias, 65536);
  cudaDeviceSynchronize();
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  cudaStream_t st;
  cudaStreamCreate(&st);
  int64_t launches = 0;
  LaunchCtx c;
  c.stream = st; c.err = err; c.launches = &launches; c.num_sms = nsm; c.host_fail = 0;
  struct Case { std::string name; GemmArgs g; };
  std::vector<Case> cs;
  auto mk = [&](const char* nm, int m, int n, int k, bool ak, int64_t lda, bool bk, int64_t ldb, int epi,
                void* out, int64_t ldo, bool of) -> GemmArgs& {
    GemmArgs g;
    memset(&g, 0, sizeof(g));
    g.M = m; g.N = n; g.K = k; g.A = A; g.lda = lda; g.a_kmajor = ak; g.B = W; g.ldb = ldb; g.b_kmajor = bk;
    g.epi = epi; g.out = out; g.ldo = ldo; g.out_f32 = of;
    g.splitk_scratch = splitk; g.splitk_scratch_floats = 16 * C * C; g.splitk_flags = flags; g.splitk_flag_count = 8192;
    cs.push_back({nm, g});
    return cs.back().g;
  };
  { GemmArgs& g = mk("qkv_fwd", M, 3 * C, C, true, C, true, C, EPI_STORE, O, 3 * C, false); g.bias = bias; }
  { GemmArgs& g = mk("attproj_fwd", M, C, C, true, C, true, C, EPI_RESIDUAL, OF, C, true); g.bias = bias; g.aux = AUXF; }
  { GemmArgs& g = mk("fc_fwd", M, 4 * C, C, true, C, true, C, EPI_GELU_FWD, O, 4 * C, false); g.bias = bias; g.out2 = O2; }
  { GemmArgs& g = mk("fcproj_fwd", M, C, 4 * C, true, 4 * C, true, 4 * C, EPI_RESIDUAL, OF, C, true); g.bias = bias; g.aux = AUXF; }
  mk("head_fwd", M, Vp, C, true, C, true, C, EPI_STORE, O, Vp, false);
  mk("head_dgrad", M, C, Vp, true, Vp, false, C, EPI_STORE, O, C, false);
  mk("head_wgrad", Vp, C, M, false, Vp, false, C, EPI_ACCUM, G, C, true);
  { GemmArgs& g = mk("fcproj_dgrad", M, 4 * C, C, true, C, false, 4 * C, EPI_MUL_AUX, O, 4 * C, false); g.aux = AUXB; g.colsum_out = colsum; }
  mk("fcproj_wgrad", C, 4 * C, M, false, C, false, 4 * C, EPI_ACCUM, G, 4 * C, true);
  mk("fc_dgrad", M, C, 4 * C, true, 4 * C, false, C, EPI_STORE, O, C, false);
  mk("fc_wgrad", 4 * C, C, M, false, 4 * C, false, C, EPI_ACCUM, G, C, true);
  { GemmArgs& g = mk("attproj_dgrad", M, C, C, true, C, false, C, EPI_DOT_AUX, O, C, false); g.aux = AUXB; g.dot_out = dsum; g.dot_T = T; }
  mk("attproj_wgrad", C, C, M, false, C, false, C, EPI_ACCUM, G, C, true);
  mk("qkv_dgrad", M, C, 3 * C, true, 3 * C, false, C, EPI_STORE, O, C, false);
  mk("qkv_wgrad", 3 * C, C, M, false, 3 * C, false, C, EPI_ACCUM, G, C, true);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  printf("{");
  double tot = 0, totf = 0;
  for (size_t i = 0; i < cs.size(); i++) {
    const GemmArgs& g = cs[i].g;
    usleep(500000);
    for (int r = 0; r < 5; r++) launch_gemm_bf16(c, g);
    cudaEventRecord(e0, st);
    for (int r = 0; r < 20; r++) launch_gemm_bf16(c, g);
    cudaEventRecord(e1, st);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    ms /= 20;
    const double fl = 2.0 * g.M * (double)g.N * g.K;
    tot += ms;
    totf += fl;
    printf("\"%s\": {\"M\": %d, \"N\": %d, \"K\": %d, \"us\": %.1f, \"tflops\": %.0f}, ", cs[i].name.c_str(), g.M, g.N,
           g.K, ms * 1e3, fl / ms / 1e9);
  }
  int herr = 0;
  const cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  printf("\"total_us\": %.1f, \"total_tflops\": %.0f, \"err\": %d, \"host_fail\": %d, \"cuda\": \"%s\"}\n", tot * 1e3,
         totf / tot / 1e9, herr, c.host_fail, cudaGetErrorString(e));
  return e == cudaSuccess && herr == 0 && c.host_fail == 0 ? 0 : 1;
}
