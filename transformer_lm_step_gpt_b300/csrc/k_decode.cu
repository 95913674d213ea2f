// k_decode.cu -- generation with a key/value cache: the attention of one new
// query row per sequence over the cached keys and values, and the draw of the
// next token from the scores of that row.
//
// GeekNews, "A GPT-2-based ChatGPT clone in 3000 bytes of C", section "How KV
// caching works": once a token has been generated, the keys and values of the
// earlier rows are kept and only the new row is computed; section "The
// Transformer core": the final LayerNorm output at the last position times the
// embedding matrix scores the candidates for the next token.  The cache is the
// per-layer qkv activation [B, T, 3C] of the forward pass: row t of sequence b
// holds [q | k | v] of position t.
#include <cuda.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"

#define DEC_THREADS 256
#define SMP_THREADS 1024

template <typename T>
__device__ __forceinline__ void load8f(const T* p, float* f);
template <>
__device__ __forceinline__ void load8f<float>(const float* p, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <>
__device__ __forceinline__ void load8f<bf16>(const bf16* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Block-wide reductions over DEC_THREADS / SMP_THREADS threads through
// shared scratch red[32]; every thread gets the result.  The order of the
// additions is fixed (lanes by shuffle tree, then warps in index order).
template <int NT>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < NT / 32; i++) r = fmaxf(r, red[i]);
  return r;
}
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < NT / 32; i++) r += red[i];
  return r;
}

__device__ __forceinline__ uint32_t dec_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void dec_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ float dec_ld_cluster(const float* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// y[b, h*hs + d] = sum_{j <= pos} p_j v_j[d],  p = softmax_j(q . k_j * scale),
// q = row pos of qkv[b] (part q), k_j / v_j = row j (parts k / v), head h.
// A cluster of KS CTAs per (b, h), CTA r taking the contiguous key range
// [r*kr, (r+1)*kr) of 0..pos: its scores (thread per key, kept in shared
// memory), their maximum m_r, sum s_r of exp(score - m_r) and the weighted
// sum o_r of the value rows (whole rows per warp load, warps added in
// order).  The first CTA of the cluster then combines the ranks in order
// through distributed shared memory: m = max m_r, y = sum_r e^(m_r - m) o_r
// / sum_r e^(m_r - m) s_r -- the softmax over all keys, split (the
// split-softmax identity), with a result that does not depend on scheduling.
template <typename T, int HS>
__global__ void __launch_bounds__(DEC_THREADS)
    attn_decode_kernel(T* y, int64_t ldy, const T* qkv, int T_, int C, int NH, const int* pos_dev, float scale,
                       int KS) {
  pdl_trigger();
  extern __shared__ float dsm[];
  constexpr int hs = HS;
  float* qs = dsm;              // [hs]
  float* red = qs + hs;         // [32]
  float* part = red + 32;       // [hs + 2]: this rank's o (hs), m, s
  float* sc = part + hs + 2;    // [kr], later the warps' partial sums (8 x hs)
  const uint32_t rank = KS > 1 ? dec_cluster_rank() : 0u;
  const int bh = blockIdx.x / KS, b = bh / NH, h = bh % NH;
  const int tid = threadIdx.x;
  const int64_t C3 = 3 * (int64_t)C;
  const T* base = qkv + (int64_t)b * T_ * C3;
  pdl_wait();
  const int pos = *pos_dev;
  const int kr = (pos + 1 + KS - 1) / KS;
  const int j0 = (int)rank * kr, j1 = min(pos + 1, j0 + kr);  // this rank's keys [j0, j1); may be empty
  for (int d = tid; d < hs; d += DEC_THREADS) qs[d] = to_f(base[(int64_t)pos * C3 + h * hs + d]);
  __syncthreads();
  float mx = -INFINITY;
  for (int j = j0 + tid; j < j1; j += DEC_THREADS) {
    const T* k = base + (int64_t)j * C3 + C + h * hs;
    float f[HS];  // the whole key row in flight at once
#pragma unroll
    for (int d = 0; d < HS; d += 8) load8f<T>(k + d, f + d);
    float s = 0.f;
#pragma unroll
    for (int d = 0; d < HS; d++) s = fmaf(qs[d], f[d], s);
    s *= scale;
    sc[j - j0] = s;
    mx = fmaxf(mx, s);
  }
  mx = block_max<DEC_THREADS>(mx, red);
  float sum = 0.f;
  for (int j = j0 + tid; j < j1; j += DEC_THREADS) {
    const float e = j1 > j0 ? expf(sc[j - j0] - mx) : 0.f;
    sc[j - j0] = e;
    sum += e;
  }
  sum = block_sum<DEC_THREADS>(sum, red);  // its barriers also publish sc[]
  // weighted sum of the values: a key's row of hs values is read by LPK =
  // hs/8 lanes (16 bytes each), so a warp reads KPW = 32/LPK whole rows per
  // load; warp w takes keys j0 + w*KPW + r*8*KPW + (lane / LPK), four rows
  // per lane in flight, and keeps 8 partial sums (its lane's 8 dimensions)
  constexpr int LPK = HS / 8, KPW = 32 / LPK;
  const int warp = tid >> 5, lane = tid & 31;
  const int kl = lane / LPK, d0 = (lane % LPK) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = 0.f;
  const T* vbase = base + 2 * C + h * hs + d0;
  const int step = (DEC_THREADS / 32) * KPW;
  int j = j0 + warp * KPW + kl;
  for (; j + 3 * step < j1; j += 4 * step) {
    float f[4][8];
#pragma unroll
    for (int u = 0; u < 4; u++) load8f<T>(vbase + (int64_t)(j + u * step) * C3, f[u]);
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float p = sc[j + u * step - j0];
#pragma unroll
      for (int i = 0; i < 8; i++) acc[i] = fmaf(p, f[u][i], acc[i]);
    }
  }
  for (; j < j1; j += step) {
    float f[8];
    load8f<T>(vbase + (int64_t)j * C3, f);
    const float p = sc[j - j0];
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = fmaf(p, f[i], acc[i]);
  }
  // add the KPW key slots of the warp (lanes with the same lane % LPK)
  for (int o = LPK; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  }
  __syncthreads();  // every thread is done reading sc[]: reuse it for the warps' sums
  if (kl == 0) {
#pragma unroll
    for (int i = 0; i < 8; i++) sc[warp * hs + d0 + i] = acc[i];
  }
  __syncthreads();
  if (tid < hs) {
    float r = 0.f;
    for (int w = 0; w < DEC_THREADS / 32; w++) r += sc[w * hs + tid];
    part[tid] = r;
  }
  if (tid == 0) { part[hs] = mx; part[hs + 1] = sum; }
  if (KS == 1) {
    __syncthreads();
    if (tid < hs) y[(int64_t)b * ldy + h * hs + tid] = from_f<T>(part[tid] / part[hs + 1]);
    return;
  }
  dec_cluster_sync();  // every rank's (o, m, s) in its shared memory
  if (rank == 0 && tid < hs) {
    float m = -INFINITY;
    for (int q = 0; q < KS; q++) m = fmaxf(m, dec_ld_cluster(part + hs, (uint32_t)q));
    float o = 0.f, l = 0.f;
    for (int q = 0; q < KS; q++) {
      const float mq = dec_ld_cluster(part + hs, (uint32_t)q);
      const float f = mq == -INFINITY ? 0.f : expf(mq - m);  // a rank without keys adds nothing
      o += f * dec_ld_cluster(part + tid, (uint32_t)q);
      l += f * dec_ld_cluster(part + hs + 1, (uint32_t)q);
    }
    y[(int64_t)b * ldy + h * hs + tid] = from_f<T>(o / l);
  }
  dec_cluster_sync();  // the first rank has read the others: they may exit
}

// The same for bf16 and head size 64, with the rank's key and value rows
// staged by TMA: one bulk tensor copy per 128 rows brings the rows [j0,
// j0 + 128 nbox) of k and of v (128-byte swizzled: logical 16-byte chunk c of
// row r sits at chunk c ^ (r & 7)) into shared memory at once, so the
// scores (thread per key) and the weighted sum (whole rows per warp) read
// shared memory instead of waiting on one global load after another.
#define DEC_ROWS 128
__global__ void __launch_bounds__(DEC_THREADS)
    attn_decode_tma_kernel(const __grid_constant__ CUtensorMap tm, bf16* y, int64_t ldy, const bf16* qkv, int T_,
                           int C, int NH, const int* pos_dev, float scale, int KS, int nbox, int* err) {
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t dtm[];
  constexpr int HS = 64;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dtm) + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = sm;                                   // [nbox * 128 rows][128 B]
  uint8_t* sV = sK + (size_t)nbox * DEC_ROWS * 128;   // same
  float* qs = reinterpret_cast<float*>(sV + (size_t)nbox * DEC_ROWS * 128);  // [64]
  float* red = qs + HS;                               // [32]
  float* part = red + 32;                             // [66]: o, m, s
  float* sc = part + HS + 2;                          // [nbox * 128], later the warps' sums [8][64]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sc + max(nbox * DEC_ROWS, (DEC_THREADS / 32) * HS));
  const uint32_t rank = KS > 1 ? dec_cluster_rank() : 0u;
  const int bh = blockIdx.x / KS, b = bh / NH, h = bh % NH;
  const int tid = threadIdx.x;
  const int64_t C3 = 3 * (int64_t)C;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm);
  }
  __syncthreads();
  pdl_wait();
  const int pos = *pos_dev;
  const int kr = (pos + 1 + KS - 1) / KS;
  const int j0 = (int)rank * kr, j1 = min(pos + 1, j0 + kr);  // this rank's keys [j0, j1); may be empty
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * nbox * DEC_ROWS * 128));
    for (int i = 0; i < nbox; i++) {
      tma_load_3d(sK + (size_t)i * DEC_ROWS * 128, &tm, bar, C + h * HS, j0 + i * DEC_ROWS, b);
      tma_load_3d(sV + (size_t)i * DEC_ROWS * 128, &tm, bar, 2 * C + h * HS, j0 + i * DEC_ROWS, b);
    }
  }
  if (tid < HS) qs[tid] = __bfloat162float(qkv[((int64_t)b * T_ + pos) * C3 + h * HS + tid]);
  __syncthreads();
  mbar_wait(bar, 0, err);
  float mx = -INFINITY;
  for (int j = j0 + tid; j < j1; j += DEC_THREADS) {
    const int r = j - j0;
    const uint8_t* row = sK + (size_t)r * 128;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; c++) {
      float f[8];
      load8f<bf16>(reinterpret_cast<const bf16*>(row + ((c ^ (r & 7)) << 4)), f);
#pragma unroll
      for (int i = 0; i < 8; i++) s = fmaf(qs[c * 8 + i], f[i], s);
    }
    s *= scale;
    sc[r] = s;
    mx = fmaxf(mx, s);
  }
  mx = block_max<DEC_THREADS>(mx, red);
  float sum = 0.f;
  for (int j = j0 + tid; j < j1; j += DEC_THREADS) {
    const float e = expf(sc[j - j0] - mx);
    sc[j - j0] = e;
    sum += e;
  }
  sum = block_sum<DEC_THREADS>(sum, red);  // its barriers also publish sc[]
  // weighted sum of the value rows: 8 lanes per row (16 bytes each), 4 rows
  // per warp step; warp w takes rows w*4 + (lane / 8) + 32 i
  const int warp = tid >> 5, lane = tid & 31;
  const int kl = lane >> 3, cl = lane & 7;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = 0.f;
  for (int r = warp * 4 + kl; r < j1 - j0; r += 32) {
    float f[8];
    load8f<bf16>(reinterpret_cast<const bf16*>(sV + (size_t)r * 128 + ((cl ^ (r & 7)) << 4)), f);
    const float p = sc[r];
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = fmaf(p, f[i], acc[i]);
  }
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  }
  __syncthreads();  // every thread is done reading sc[]: reuse it for the warps' sums
  if (kl == 0) {
#pragma unroll
    for (int i = 0; i < 8; i++) sc[warp * HS + cl * 8 + i] = acc[i];
  }
  __syncthreads();
  if (tid < HS) {
    float r = 0.f;
    for (int w = 0; w < DEC_THREADS / 32; w++) r += sc[w * HS + tid];
    part[tid] = r;
  }
  if (tid == 0) { part[HS] = mx; part[HS + 1] = sum; }
  if (KS == 1) {
    __syncthreads();
    if (tid < HS) y[(int64_t)b * ldy + h * HS + tid] = __float2bfloat16_rn(part[tid] / part[HS + 1]);
    return;
  }
  dec_cluster_sync();  // every rank's (o, m, s) in its shared memory
  if (rank == 0 && tid < HS) {
    float m = -INFINITY;
    for (int q = 0; q < KS; q++) m = fmaxf(m, dec_ld_cluster(part + HS, (uint32_t)q));
    float o = 0.f, l = 0.f;
    for (int q = 0; q < KS; q++) {
      const float mq = dec_ld_cluster(part + HS, (uint32_t)q);
      const float f = mq == -INFINITY ? 0.f : expf(mq - m);  // a rank without keys adds nothing
      o += f * dec_ld_cluster(part + tid, (uint32_t)q);
      l += f * dec_ld_cluster(part + HS + 1, (uint32_t)q);
    }
    y[(int64_t)b * ldy + h * HS + tid] = __float2bfloat16_rn(o / l);
  }
  dec_cluster_sync();  // the first rank has read the others: they may exit
}

template <typename T>
void launch_attention_decode(LaunchCtx& c, T* y, int64_t ldy, const T* qkv, int B, int T_, int C, int NH,
                             const int* pos) {
  const int hs = C / NH;
  // split the keys over a cluster of up to 8 CTAs (fixed by the cache size,
  // so that the launch does not depend on the position)
  const int KS = std::max(1, std::min(8, (T_ + 63) / 64));
  const int kr = (T_ + KS - 1) / KS;  // the most keys a rank can get
  const float scale = 1.f / sqrtf((float)hs);
  if constexpr (sizeof(T) == 2) {
    if (hs == 64) {  // key / value rows staged by TMA
      CUtensorMap tmap;
      if (!attn_tmap_btw(&tmap, qkv, B, T_, 3 * C, DEC_ROWS)) {
        c.host_fail = 1;
        return;
      }
      const int nbox = (kr + DEC_ROWS - 1) / DEC_ROWS;
      const size_t smem = 1024 + (size_t)2 * nbox * DEC_ROWS * 128 +
                          sizeof(float) * (64 + 32 + 66 + std::max(nbox * DEC_ROWS, (DEC_THREADS / 32) * 64)) + 8;
      static bool attr = false;
      if (!attr) {
        cudaFuncSetAttribute(attn_decode_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        attr = true;
      }
      if (KS > 1)
        launch_pdl_cluster(c, attn_decode_tma_kernel, dim3(B * NH * KS), dim3(DEC_THREADS), smem, KS, tmap, y, ldy,
                           qkv, T_, C, NH, pos, scale, KS, nbox, c.err);
      else
        launch_pdl(c, attn_decode_tma_kernel, dim3(B * NH), dim3(DEC_THREADS), smem, tmap, y, ldy, qkv, T_, C, NH,
                   pos, scale, KS, nbox, c.err);
      return;
    }
  }
  const size_t smem = sizeof(float) * (hs + 32 + hs + 2 + std::max(kr, (DEC_THREADS / 32) * hs));
  auto kern = hs == 16 ? attn_decode_kernel<T, 16>
              : hs == 32 ? attn_decode_kernel<T, 32>
              : hs == 64 ? attn_decode_kernel<T, 64>
                         : attn_decode_kernel<T, 128>;
  if (KS > 1)
    launch_pdl_cluster(c, kern, dim3(B * NH * KS), dim3(DEC_THREADS), smem, KS, y, ldy, qkv, T_, C, NH, pos, scale,
                       KS);
  else
    launch_pdl(c, kern, dim3(B * NH), dim3(DEC_THREADS), smem, y, ldy, qkv, T_, C, NH, pos, scale, KS);
}
template void launch_attention_decode<float>(LaunchCtx&, float*, int64_t, const float*, int, int, int, int, const int*);
template void launch_attention_decode<bf16>(LaunchCtx&, bf16*, int64_t, const bf16*, int, int, int, int, const int*);

// One CTA per row b of logits [B, ld]: the next token from the first V
// scores (inverse-CDF sampling of the softmax at `temperature` with the
// uniform draw u[b]; temperature <= 0: the first index of the largest score).
// Thread t owns the contiguous chunk [t*cs, (t+1)*cs) of the row; the chunk
// sums of e_i = exp((l_i - max) / temperature) are scanned in thread order,
// and the thread whose chunk holds the threshold u * sum walks it again.
template <typename T>
__global__ void __launch_bounds__(SMP_THREADS)
    sample_kernel(int32_t* next, const T* logits, int64_t ld, int V, const float* temp_dev, const float* u) {
  pdl_trigger();
  __shared__ float red[32];
  __shared__ float wsum[SMP_THREADS / 32];
  __shared__ int pick;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const T* l = logits + (int64_t)b * ld;
  pdl_wait();
  const float temperature = *temp_dev;
  const int cs = (V + SMP_THREADS - 1) / SMP_THREADS;
  const int i0 = min(tid * cs, V), i1 = min(i0 + cs, V);
  // largest score; its first index
  float mx = -INFINITY;
  int arg = INT_MAX;
  for (int i = i0; i < i1; i++) {
    const float x = to_f(l[i]);
    if (x > mx) { mx = x; arg = i; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mx, o);
    const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
    if (om > mx || (om == mx && oa < arg)) { mx = om; arg = oa; }
  }
  __shared__ int rarg[32];
  if (lane == 0) { red[w] = mx; rarg[w] = arg; }
  __syncthreads();
  if (tid == 0) {
    float bm = red[0];
    int ba = rarg[0];
    for (int i = 1; i < SMP_THREADS / 32; i++)
      if (red[i] > bm || (red[i] == bm && rarg[i] < ba)) { bm = red[i]; ba = rarg[i]; }
    red[0] = bm;
    pick = ba;
  }
  __syncthreads();
  if (!(temperature > 0.f)) {
    if (tid == 0) next[b] = pick;
    return;
  }
  const float m = red[0], it = 1.f / temperature;
  float s = 0.f;
  int lastnz = -1;
  for (int i = i0; i < i1; i++) {
    const float e = expf((to_f(l[i]) - m) * it);
    s += e;
    if (e > 0.f) lastnz = i;
  }
  // inclusive scan of the chunk sums in thread order
  float incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[w] = incl;
  int lnz = lastnz;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lnz = max(lnz, __shfl_xor_sync(0xffffffffu, lnz, o));
  __syncthreads();
  if (tid == 0) {
    float run = 0.f;
    for (int i = 0; i < SMP_THREADS / 32; i++) {
      const float t = wsum[i];
      wsum[i] = run;  // exclusive prefix of warp i
      run += t;
    }
    red[1] = run;  // total
  }
  if (lane == 0) rarg[w] = lnz;
  __syncthreads();
  if (tid == 0) {
    int g = -1;
    for (int i = 0; i < SMP_THREADS / 32; i++) g = max(g, rarg[i]);
    pick = g;  // fallback: the last index with a nonzero weight
  }
  __syncthreads();
  const float total = red[1];
  const float target = u[b] * total;
  __shared__ float excl_s[SMP_THREADS];
  excl_s[tid] = wsum[w] + (incl - s);  // sum of the chunks before this thread's
  __syncthreads();
  // thread t claims the threshold when excl[t] <= target < excl[t+1]
  // (excl[SMP_THREADS] = +inf): at least one thread does, since excl[0] = 0;
  // if rounding lets two claim, the smaller index wins; a claimed chunk
  // whose running sum never passes the threshold (rounding again) yields
  // its last index with a nonzero weight.  Otherwise (the threshold at the
  // very top) the last index with a nonzero weight overall is kept.
  const float ex = excl_s[tid];
  const float ex_next = tid + 1 < SMP_THREADS ? excl_s[tid + 1] : INFINITY;
  if (s > 0.f && ex <= target && target < ex_next) {
    float run = ex;
    int found = lastnz;
    for (int i = i0; i < i1; i++) {
      run += expf((to_f(l[i]) - m) * it);
      if (run > target) { found = i; break; }
    }
    atomicMin(&pick, found);
  }
  __syncthreads();
  if (tid == 0) next[b] = pick;
}

template <typename T>
void launch_sample(LaunchCtx& c, int32_t* next, const T* logits, int64_t ld, int B, int V, const float* temperature,
                   const float* u) {
  launch_pdl(c, sample_kernel<T>, dim3(B), dim3(SMP_THREADS), 0, next, logits, ld, V, temperature, u);
}
template void launch_sample<float>(LaunchCtx&, int32_t*, const float*, int64_t, int, int, const float*, const float*);
template void launch_sample<bf16>(LaunchCtx&, int32_t*, const bf16*, int64_t, int, int, const float*, const float*);

// x[b, :] = wte[tok[b], :] + wpe[pos, :]: one CTA per row, C/4 threads.
__global__ void decode_embed_kernel(float* x, const int32_t* tok, const float* wte, const float* wpe,
                                    const int* pos_dev, int C, int V, int* err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  int id = tok[b];
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) record_error(err, DEVERR_TOKEN);
    id = 0;
  }
  const int pos = *pos_dev;
  for (int c4 = threadIdx.x; c4 < C / 4; c4 += blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(wte + (int64_t)id * C)[c4];
    const float4 e = reinterpret_cast<const float4*>(wpe + (int64_t)pos * C)[c4];
    reinterpret_cast<float4*>(x + (int64_t)b * C)[c4] = make_float4(a.x + e.x, a.y + e.y, a.z + e.z, a.w + e.w);
  }
}

void launch_decode_embed(LaunchCtx& c, float* x, const int32_t* tok, const float* wte, const float* wpe,
                         const int* pos, int B, int C, int V) {
  launch_pdl(c, decode_embed_kernel, dim3(B), dim3(std::min(256, C / 4)), 0, x, tok, wte, wpe, pos, C, V, c.err);
}

__global__ void decode_inputs_kernel(int32_t* tok_dst, const int32_t* tok_src, float* u_dst, const float* u_src,
                                     int* pos_dst, int pos, float* temp_dst, float temperature, int B) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    tok_dst[i] = tok_src[i];
    u_dst[i] = u_src[i];
  }
  if (threadIdx.x == 0) {
    *pos_dst = pos;
    *temp_dst = temperature;
  }
}

void launch_decode_inputs(LaunchCtx& c, int32_t* tok_dst, const int32_t* tok_src, float* u_dst, const float* u_src,
                          int* pos_dst, int pos, float* temp_dst, float temperature, int B) {
  launch_pdl(c, decode_inputs_kernel, dim3(1), dim3(128), 0, tok_dst, tok_src, u_dst, u_src, pos_dst, pos, temp_dst,
             temperature, B);
}
