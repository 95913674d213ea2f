// k_fp8.cu -- lower-precision matmuls: E4M3 (8-bit float) operands with
// per-tensor scaling.
//
// QbitAI, "OpenAI founder hand-writes a thousand lines of C to train GPT",
// names lowering the precision from fp32 to fp16 or lower as a next step.
// Here an operand x is stored as E4M3 codes q = E4M3(x * s) with one scale
// s = 448 / max|x| per tensor (the largest magnitude lands on the largest
// code), and a matmul of two such operands accumulates the code products in
// fp32 on the tensor cores (tcgen05 kind::f8f6f4, twice the bf16 rate) and
// divides by s_a * s_b in its epilogue.
#include <algorithm>
#include <cstdint>

#include "../../include/gpt2.h"
#include "common.cuh"
#include "kernels.h"

// max|x| into *amax (as float bits: for non-negative floats the unsigned
// order is the numeric order, so atomicMax gives the same result whatever
// the order of the updates).  NaN entries are skipped.
template <typename T>
__global__ void fp8_amax_kernel(const T* x, int64_t n, float* amax) {
  pdl_trigger();
  pdl_wait();
  float m = 0.f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = fabsf(to_f(x[i]));
    if (!isnan(v)) m = fmaxf(m, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(m));
}

// two codes: lo from a, hi from b (round to nearest even, saturating)
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// q[i] = E4M3(x[i] * s), s = 448 / scale[1] (1 if scale[1] is 0); scale[0] = s.
// Eight values per thread per step (one 8-byte store).
template <typename T>
__global__ void fp8_quantize_kernel(const T* x, int64_t n, float* scale, uint8_t* q) {
  pdl_trigger();
  pdl_wait();
  const float amax = scale[1];
  const float s = amax > 0.f ? 448.f / amax : 1.f;
  if (blockIdx.x == 0 && threadIdx.x == 0) scale[0] = s;
  const int64_t n8 = n / 8;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] = to_f(x[i * 8 + j]) * s;
    uint2 w;
    w.x = (uint32_t)e4m3x2(v[0], v[1]) | ((uint32_t)e4m3x2(v[2], v[3]) << 16);
    w.y = (uint32_t)e4m3x2(v[4], v[5]) | ((uint32_t)e4m3x2(v[6], v[7]) << 16);
    reinterpret_cast<uint2*>(q)[i] = w;
  }
  // the n % 8 tail
  const int64_t t = n8 * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t < n) q[t] = (uint8_t)(e4m3x2(to_f(x[t]) * s, 0.f) & 0xff);
}

void launch_fp8_quantize(LaunchCtx& c, const void* x, bool x_bf16, int64_t n, uint8_t* q, float* scale) {
  cudaMemsetAsync(scale + 1, 0, sizeof(float), c.stream);
  const int grid = (int)std::min<int64_t>((n / 8 + 255) / 256 + 1, (int64_t)std::max(c.num_sms, 1) * 8);
  if (x_bf16) {
    launch_pdl(c, fp8_amax_kernel<bf16>, dim3(grid), dim3(256), 0, static_cast<const bf16*>(x), n, scale + 1);
    launch_pdl(c, fp8_quantize_kernel<bf16>, dim3(grid), dim3(256), 0, static_cast<const bf16*>(x), n, scale, q);
  } else {
    launch_pdl(c, fp8_amax_kernel<float>, dim3(grid), dim3(256), 0, static_cast<const float*>(x), n, scale + 1);
    launch_pdl(c, fp8_quantize_kernel<float>, dim3(grid), dim3(256), 0, static_cast<const float*>(x), n, scale, q);
  }
}

// ---------------------------------------------------------------- C ABI
// The error word of these model-less entry points (bounded waits), one per
// device; gpt2_fp8_check reads and clears it.
static __device__ int g_fp8_err;

static int* fp8_err_word() {
  static int* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fp8_err) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

static LaunchCtx fp8_ctx(void* stream, int64_t* launches) {
  LaunchCtx c;
  c.stream = static_cast<cudaStream_t>(stream);
  c.err = fp8_err_word();
  c.launches = launches;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  c.num_sms = sms;
  c.host_fail = 0;
  return c;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" int gpt2_fp8_quantize(const void* x, int32_t x_is_bf16, int64_t n, uint8_t* q, float* scale,
                                 void* cuda_stream) {
  if (!x || !q || !scale || n < 1) {
    set_global_error("gpt2_fp8_quantize: NULL pointer or n < 1");
    return GPT2_ERR_ARG;
  }
  if (!aligned16(x) || !aligned16(q)) {
    set_global_error("gpt2_fp8_quantize: x and q must be 16-byte aligned");
    return GPT2_ERR_ARG;
  }
  int64_t launches = 0;
  LaunchCtx c = fp8_ctx(cuda_stream, &launches);
  launch_fp8_quantize(c, x, x_is_bf16 != 0, n, q, scale);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || c.host_fail) {
    set_global_error(e != cudaSuccess ? cudaGetErrorString(e) : "gpt2_fp8_quantize: launch failed");
    return GPT2_ERR_CUDA;
  }
  return GPT2_OK;
}

extern "C" int gpt2_fp8_matmul(const uint8_t* a, int64_t lda, const float* scale_a, const uint8_t* b, int64_t ldb,
                               const float* scale_b, int32_t M, int32_t N, int32_t K, const float* bias, void* out,
                               int64_t ldo, int32_t out_is_bf16, void* cuda_stream) {
  if (!a || !b || !scale_a || !scale_b || !out || M < 1 || N < 1 || K < 1) {
    set_global_error("gpt2_fp8_matmul: NULL pointer or a size below 1");
    return GPT2_ERR_ARG;
  }
  const int64_t esz = out_is_bf16 ? 2 : 4;
  if (lda < K || ldb < K || lda % 16 || ldb % 16 || ldo < N || (ldo * esz) % 16 || !aligned16(a) || !aligned16(b) ||
      !aligned16(out) || (bias && !aligned16(bias))) {
    set_global_error("gpt2_fp8_matmul: need lda, ldb >= K and multiples of 16, ldo >= N with 16-byte rows, "
                     "16-byte aligned a, b, out and bias");
    return GPT2_ERR_ARG;
  }
  if (!gemm_bf16_init()) {
    set_global_error("gpt2_fp8_matmul: the driver's tensor-map encoder is unavailable");
    return GPT2_ERR_CUDA;
  }
  int64_t launches = 0;
  LaunchCtx c = fp8_ctx(cuda_stream, &launches);
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.M = M; g.N = N; g.K = K;
  g.A = a; g.lda = lda; g.a_kmajor = true;
  g.B = b; g.ldb = ldb; g.b_kmajor = true;
  g.epi = EPI_STORE; g.out = out; g.ldo = ldo; g.out_f32 = !out_is_bf16;
  g.bias = bias;
  g.dequant_a = scale_a;
  g.dequant_b = scale_b;
  launch_gemm_fp8(c, g);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || c.host_fail) {
    set_global_error(e != cudaSuccess ? cudaGetErrorString(e) : "gpt2_fp8_matmul: launch failed");
    return GPT2_ERR_CUDA;
  }
  return GPT2_OK;
}

extern "C" int gpt2_fp8_check(void* cuda_stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  int* w = fp8_err_word();
  int v = 0;
  if (e == cudaSuccess && w) e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess || !w) {
    set_global_error(e != cudaSuccess ? cudaGetErrorString(e) : "gpt2_fp8_check: no error word");
    return GPT2_ERR_CUDA;
  }
  if (v) {
    cudaMemset(w, 0, sizeof(int));
    set_global_error("gpt2_fp8_check: a bounded device wait expired");
    return GPT2_ERR_TIMEOUT;
  }
  return GPT2_OK;
}
