// Tensor-pipe rate probe for the attention and matmul kernels' design:
// cycles per tcgen05.mma (K = 16, bf16) by shape, and the same stream of
// MMAs while other warps of the CTA run FFMA chains or packed f32x2 FMA
// chains on the issuing thread's scheduler or on the other three.
// Prints one JSON object.  Every wait is bounded (common.cuh); the busy
// warps stop on a shared flag or after a fixed count.
#include <cstdio>
#include <cstdlib>

#include "../../transformer_lm_step_gpt_b300/csrc/common.cuh"

__device__ __forceinline__ uint8_t* al1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}
#define SMEM_BYTES (1024 + 16384 + 32768 + 1024)

// one thread issues `iters` x 4 MMAs (M = 128, N, K = 16, A in smem or in
// TMEM, B K-major in smem), alternating two accumulators; warps whose bit
// is set in `busy` run FFMA (mode 1) or f32x2 FMA (mode 2) chains meanwhile
template <int N, bool TS>
__global__ void __launch_bounds__(544, 1) probe_cg1(int iters, int mode, unsigned busy, long long* out, int* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = al1024(raw);
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  __shared__ volatile int stop;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = 0x3c003c00u ^ (uint32_t)(i * 2654435761u & 0x00ff00ffu);
  if (threadIdx.x == 0) { mbar_init(&bar, 1); fence_mbar_init(); stop = 0; }
  if (warp == 0) { tmem_alloc(&slot, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = slot;
  if (warp < 4) {  // A operand words in TMEM columns 256..287
    uint32_t v[16];
    for (int i = 0; i < 16; i++) v[i] = 0x3c003c00u;
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    tmem_st16(tm + lb + 256, v);
    tmem_st16(tm + lb + 272, v);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 16) {
    if (lane == 0) {
      const uint32_t idesc = tc_idesc_bf16(128, N, false, false);
      const uint32_t a0 = smem_u32(sm), b0 = a0 + 16384;
      const long long t0 = clock64();
      for (int i = 0; i < iters; i++) {
        const uint32_t acc = tm + (uint32_t)((i & 1) * N);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
          const uint64_t bd = sw128_desc(b0 + kk * 32, 16, 1024);
          if (TS) tc_mma_bf16_ts(acc, tm + 256 + kk * 8, bd, idesc, (kk > 0 || i >= 2) ? 1u : 0u);
          else tc_mma_bf16(acc, sw128_desc(a0 + kk * 32, 16, 1024), bd, idesc, (kk > 0 || i >= 2) ? 1u : 0u);
        }
      }
      tc_commit(&bar);
      mbar_wait(&bar, 0, err);
      out[0] = clock64() - t0;
      stop = 1;
    }
  } else if ((busy >> warp) & 1u) {
    float a[8];
    for (int i = 0; i < 8; i++) a[i] = 0.001f * (threadIdx.x + i);
    for (int n = 0; !stop && n < 200000; n++) {
      if (mode == 1) {
#pragma unroll
        for (int r = 0; r < 16; r++)
#pragma unroll
          for (int i = 0; i < 8; i++) a[i] = fmaf(a[i], 0.999f, 0.001f);
      } else {
        uint64_t b2[4];
        for (int i = 0; i < 4; i++) b2[i] = f2_pack(a[2 * i], a[2 * i + 1]);
#pragma unroll
        for (int r = 0; r < 16; r++)
#pragma unroll
          for (int i = 0; i < 4; i++) b2[i] = f2_fma(b2[i], f2_pack(0.999f, 0.999f), f2_pack(0.001f, 0.001f));
        for (int i = 0; i < 4; i++) f2_unpack(b2[i], a[2 * i], a[2 * i + 1]);
      }
    }
    float s = 0.f;
    for (int i = 0; i < 8; i++) s += a[i];
    if (s == 12345.f) out[1] = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

// a CTA pair issues M = 256 MMAs (cta_group::2) from the even CTA
template <int N>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) probe_cg2(int iters, long long* out, int* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = al1024(raw);
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  const uint32_t rank = cluster_rank();
  for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += 128)
    reinterpret_cast<uint32_t*>(sm)[i] = 0x3c003c00u ^ (uint32_t)(i * 2654435761u & 0x00ff00ffu);
  if (threadIdx.x == 0) { mbar_init(&bar, 1); fence_mbar_init(); }
  if (threadIdx.x < 32) { tmem_alloc_pair(&slot, 512); tmem_relinquish_pair(); }
  fence_proxy_async_smem();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tm = slot;
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    if (rank == 0) {
      const uint32_t idesc = tc_idesc_bf16(256, N, false, false);
      const uint32_t a0 = smem_u32(sm), b0 = a0 + 16384;
      for (int i = 0; i < iters; i++) {
        const uint32_t acc = tm + (uint32_t)((i & 1) * N);
#pragma unroll
        for (int kk = 0; kk < 4; kk++)
          tc_mma_bf16_pair(acc, sw128_desc(a0 + kk * 32, 16, 1024), sw128_desc(b0 + kk * 32, 16, 1024), idesc,
                           (kk > 0 || i >= 2) ? 1u : 0u);
      }
      tc_commit_pair_both(&bar);
    }
    mbar_wait(&bar, 0, err);
    if (rank == 0) out[0] = clock64() - t0;
  }
  tc_fence_before();
  cluster_sync();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc_pair(tm, 512); }
}

static long long* g_out;
static int* g_err;
template <typename K>
static double cycles_cg1(K kern, int mode, unsigned busy) {
  const int iters = 256;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  for (int rep = 0; rep < 2; rep++) kern<<<1, 544, SMEM_BYTES>>>(iters, mode, busy, g_out, g_err);
  if (cudaDeviceSynchronize() != cudaSuccess) { printf("{\"error\": \"launch\"}\n"); exit(1); }
  long long h = 0;
  cudaMemcpy(&h, g_out, sizeof(long long), cudaMemcpyDeviceToHost);
  return h / (iters * 4.0);
}
template <typename K>
static double cycles_cg2(K kern) {
  const int iters = 256;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  for (int rep = 0; rep < 2; rep++) kern<<<2, 128, SMEM_BYTES>>>(iters, g_out, g_err);
  if (cudaDeviceSynchronize() != cudaSuccess) { printf("{\"error\": \"launch\"}\n"); exit(1); }
  long long h = 0;
  cudaMemcpy(&h, g_out, sizeof(long long), cudaMemcpyDeviceToHost);
  return h / (iters * 4.0);
}

int main() {
  cudaMalloc(&g_out, 2 * sizeof(long long));
  cudaMalloc(&g_err, sizeof(int));
  cudaMemset(g_err, 0, sizeof(int));
  // busy warps: 0x1111 = warps 0, 4, 8, 12 (the issuing warp 16's scheduler);
  // 0xeeee = the 12 warps on the other three schedulers
  printf("{\"cg1_ss_n64\": %.1f, \"cg1_ss_n128\": %.1f, \"cg1_ss_n256\": %.1f, \"cg1_ts_n64\": %.1f, "
         "\"cg1_ts_n128\": %.1f, \"cg2_n64\": %.1f, \"cg2_n128\": %.1f, \"cg2_n256\": %.1f, "
         "\"ts_n64_ffma_same_scheduler\": %.1f, \"ts_n64_ffma_other_schedulers\": %.1f, "
         "\"ts_n64_f32x2_same_scheduler\": %.1f",
         cycles_cg1(probe_cg1<64, false>, 0, 0u), cycles_cg1(probe_cg1<128, false>, 0, 0u),
         cycles_cg1(probe_cg1<256, false>, 0, 0u), cycles_cg1(probe_cg1<64, true>, 0, 0u),
         cycles_cg1(probe_cg1<128, true>, 0, 0u), cycles_cg2(probe_cg2<64>), cycles_cg2(probe_cg2<128>),
         cycles_cg2(probe_cg2<256>), cycles_cg1(probe_cg1<64, true>, 1, 0x1111u),
         cycles_cg1(probe_cg1<64, true>, 1, 0xeeeeu), cycles_cg1(probe_cg1<64, true>, 2, 0x1111u));
  int err = 0;
  cudaMemcpy(&err, g_err, sizeof(int), cudaMemcpyDeviceToHost);
  printf(", \"wait_error\": %d}\n", err);
  return 0;
}
