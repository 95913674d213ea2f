// k_misc.cu -- the bandwidth-bound kernels of the step.
//
//  - parameter initialisation (Philox4x32-10 + Box-Muller, on the device)
//  - encoder forward / backward (token + position embedding; InfoQ's layer
//    list "encoder")
//  - LayerNorm forward / backward (QbitAI's worked example; GeekNews,
//    "Implementing the neural-network layers")
//  - bias-gradient column sums, fused softmax + cross-entropy (InfoQ's
//    layer list), mean loss, AdamW (InfoQ: "Adam lr 1e-4")
//
// All of them are HBM-bound: each reads its inputs once with 16-byte vector
// loads, reduces rows with warp shuffles and writes its outputs once.  Every
// reduction runs in a fixed order, so results repeat bit for bit.
#include <cstdio>

#include "../../include/gpt2.h"
#include "common.cuh"
#include "kernels.h"

#define LAUNCH_CHECK(c) \
  do { (*(c).launches)++; } while (0)

static inline int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// ============================================================ init
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; r++) {
    if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
    const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
  }
}

__global__ void init_params_kernel(float* p, InitSpec s) {
  pdl_trigger();
  pdl_wait();
  const int64_t total = s.off[16];
  const double sd = 0.02, sdr = 0.02 / sqrt(2.0 * (double)(s.L > 0 ? s.L : 1));
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    int t = 0;
    while (t < 15 && e >= s.off[t + 1]) t++;
    // tensor ids: 0 wte 1 wpe 2 ln1w 3 ln1b 4 qkvw 5 qkvb 6 attprojw 7 attprojb
    //             8 ln2w 9 ln2b 10 fcw 11 fcb 12 fcprojw 13 fcprojb 14 lnfw 15 lnfb
    double scale = 0.0;
    bool draw = false;
    if (t == 0) { draw = (e - s.off[0]) / s.C < s.V; scale = sd; }
    else if (t == 1 || t == 4 || t == 10) { draw = true; scale = sd; }
    else if (t == 6 || t == 12) { draw = true; scale = sdr; }
    float v = (t == 2 || t == 8 || t == 14) ? 1.f : 0.f;
    if (draw) {
      const uint64_t pair = (uint64_t)e >> 1;
      uint32_t c[4] = {(uint32_t)pair, (uint32_t)(pair >> 32), 0u, 0u};
      philox4x32_10(c, (uint32_t)s.seed, (uint32_t)(s.seed >> 32));
      const double u1 = ((double)c[0] + 1.0) / 4294967296.0;
      const double u2 = (double)c[1] / 4294967296.0;
      const double r = sqrt(-2.0 * log(u1));
      const double th = 6.283185307179586476925 * u2;
      v = (float)(scale * ((e & 1) ? r * sin(th) : r * cos(th)));
    }
    p[e] = v;
  }
}

void launch_init_params(LaunchCtx& c, float* params, const InitSpec& s) {
  launch_pdl(c, init_params_kernel, dim3(c.num_sms * 8), dim3(256), 0, params, s);
}

__global__ void f32_to_bf16_kernel(bf16* out, const float* in, int64_t n) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = __float2bfloat16_rn(in[i]);
}
void launch_f32_to_bf16(LaunchCtx& c, bf16* out, const float* in, int64_t n) {
  launch_pdl(c, f32_to_bf16_kernel, dim3(c.num_sms * 8), dim3(256), 0, out, in, n);
}

// ============================================================ encoder
__global__ void encoder_fwd_kernel(float* out, const int32_t* tok, const float* wte,
                                   const float* wpe, int B, int T, int C, int V, int* err) {
  pdl_trigger();
  pdl_wait();
  const int C4 = C / 4;
  const int64_t n = (int64_t)B * T * C4;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / C4;
    const int c4 = (int)(idx % C4);
    const int t = (int)(i % T);
    int id = tok[i];
    if (id < 0 || id >= V) {
      if (c4 == 0) record_error(err, DEVERR_TOKEN);
      id = 0;
    }
    const float4 a = reinterpret_cast<const float4*>(wte + (int64_t)id * C)[c4];
    const float4 b = reinterpret_cast<const float4*>(wpe + (int64_t)t * C)[c4];
    reinterpret_cast<float4*>(out + i * C)[c4] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
  }
}

void launch_encoder_fwd(LaunchCtx& c, float* out, const int32_t* tok, const float* wte,
                        const float* wpe, int B, int T, int C, int V) {
  const int64_t n = (int64_t)B * T * (C / 4);
  int grid = (int)std::min<int64_t>(cdiv(n, 256), (int64_t)c.num_sms * 16);
  launch_pdl(c, encoder_fwd_kernel, dim3(grid), dim3(256), 0, out, tok, wte, wpe, B, T, C, V, c.err);
}

// dwpe[t, c] += sum_b dout[b, t, c], b in order.
__global__ void encoder_bwd_wpe_kernel(float* dwpe, const float* dout, int B, int T, int C) {
  pdl_trigger();
  pdl_wait();
  const int64_t n = (int64_t)T * C;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(idx / C), ch = (int)(idx % C);
    float s = 0.f;
#pragma unroll 8
    for (int b = 0; b < B; b++) s += __ldg(dout + ((int64_t)b * T + t) * C + ch);  // loads issued ahead, added in b order
    dwpe[idx] += s;
  }
}

// Sort the keys tok*M + position by token, stably (positions come in
// increasing order, so equal tokens end up adjacent in position order):
// one block, a least-significant-digit radix sort on the token in two
// passes of 9 bits (tokens below 2^18).  In each pass warp w owns the
// contiguous items [w*S, (w+1)*S) and walks them 32 at a time:
//   1. per-warp digit counts (__match_any_sync groups the lanes of a digit);
//   2. one exclusive scan over (digit, warp) in digit-major order gives each
//      warp's first destination per digit;
//   3. the same walk scatters each key to its warp's next slot for its
//      digit (rank among equal digits of the round = lanes below it).
// keys in `a`, the first pass writes `b`, the second writes `a` back.
#define ES_THREADS 1024
#define ES_WARPS (ES_THREADS / 32)
#define ES_BITS 9
#define ES_BINS (1 << ES_BITS)
#define ES_MAX_ROUNDS 32  // 32 x 32 items per warp: M <= 32768
__global__ void __launch_bounds__(ES_THREADS, 1)
    encoder_sort_kernel(uint32_t* a, uint32_t* b, const int32_t* tok, int M, int Vp) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int es_cnt[];  // [ES_BINS][ES_WARPS], digit-major
  __shared__ int es_sums[ES_THREADS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < M; i += ES_THREADS) {
    int id = tok[i];
    id = id < 0 ? 0 : (id >= Vp ? Vp - 1 : id);
    a[i] = (uint32_t)id * (uint32_t)M + (uint32_t)i;
  }
  __syncthreads();
  const int S = (M + ES_WARPS - 1) / ES_WARPS;  // <= 1024 items per warp (M <= 32768)
  const int w0 = warp * S, w1 = min(M, w0 + S);
  const uint32_t lt = (1u << lane) - 1u;
  for (int pass = 0; pass < 2; pass++) {
    const uint32_t* src = pass ? b : a;
    uint32_t* dst = pass ? a : b;
    const int shift = pass * ES_BITS;
    // the warp's keys in registers: round r's key of lane l is item w0 + 32r + l
    uint32_t key[ES_MAX_ROUNDS];
#pragma unroll
    for (int r = 0; r < ES_MAX_ROUNDS; r++) {
      const int i = w0 + 32 * r + lane;
      key[r] = i < w1 ? src[i] : 0xFFFFFFFFu;
    }
    for (int i = threadIdx.x; i < ES_BINS * ES_WARPS; i += ES_THREADS) es_cnt[i] = 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < ES_MAX_ROUNDS; r++) {
      if (w0 + 32 * r >= w1) break;  // warp-uniform
      const bool on = w0 + 32 * r + lane < w1;
      const uint32_t d = on ? ((key[r] / (uint32_t)M) >> shift) & (ES_BINS - 1) : 0xFFFFFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (on && (peers & lt) == 0) es_cnt[d * ES_WARPS + warp] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // exclusive scan of the ES_BINS * ES_WARPS counts, 16 per thread
    {
      constexpr int PER = ES_BINS * ES_WARPS / ES_THREADS;
      int run = 0;
#pragma unroll
      for (int k = 0; k < PER; k++) run += es_cnt[threadIdx.x * PER + k];
      es_sums[threadIdx.x] = run;
      __syncthreads();
      for (int off = 1; off < ES_THREADS; off <<= 1) {  // inclusive scan of the thread totals
        const int t = threadIdx.x >= off ? es_sums[threadIdx.x - off] : 0;
        __syncthreads();
        es_sums[threadIdx.x] += t;
        __syncthreads();
      }
      int base = es_sums[threadIdx.x] - run;
#pragma unroll
      for (int k = 0; k < PER; k++) {
        const int v = es_cnt[threadIdx.x * PER + k];
        es_cnt[threadIdx.x * PER + k] = base;
        base += v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < ES_MAX_ROUNDS; r++) {
      if (w0 + 32 * r >= w1) break;
      const bool on = w0 + 32 * r + lane < w1;
      const uint32_t d = on ? ((key[r] / (uint32_t)M) >> shift) & (ES_BINS - 1) : 0xFFFFFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (on) {
        const int base = es_cnt[d * ES_WARPS + warp];
        dst[base + __popc(peers & lt)] = key[r];
      }
      __syncwarp();
      if (on && (peers & lt) == 0) es_cnt[d * ES_WARPS + warp] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
  }
}

__device__ __forceinline__ int lower_bound_u32(const uint32_t* a, int n, uint32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

#define ENC_PIECE 64
#define ENC_RANGE 64  // sorted indices per block
// Block b looks at the sorted indices [64b, 64b+64): those that start a
// piece (a segment start, or 64 rows into a segment) sum their piece's rows
// in order, one warp per piece.  Single-piece segments add straight into
// dwte; longer ones leave a partial per piece.
__global__ void encoder_bwd_piece_kernel(float* dwte, float* partial, const float* dout,
                                         const uint32_t* sorted, int M, int C) {
  pdl_trigger();
  pdl_wait();
  __shared__ int starts[ENC_RANGE];
  __shared__ int seg_lo[ENC_RANGE], seg_hi[ENC_RANGE];
  __shared__ int nstart;
  const int i0 = blockIdx.x * ENC_RANGE;
  if (threadIdx.x == 0) nstart = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    for (int k = threadIdx.x; k < ENC_RANGE; k += 32) {  // two rounds of 32, in index order
      const int i = i0 + k;
      bool is_start = false;
      int s0 = 0, s1 = 0;
      if (i < M) {
        const uint32_t id = sorted[i] / (uint32_t)M;
        s0 = lower_bound_u32(sorted, M, id * (uint32_t)M);
        is_start = (i - s0) % ENC_PIECE == 0;
        if (is_start) s1 = lower_bound_u32(sorted, M, (id + 1) * (uint32_t)M);
      }
      const uint32_t ball = __ballot_sync(0xffffffffu, is_start);
      const int slot = nstart + __popc(ball & ((1u << threadIdx.x) - 1u));
      if (is_start) {
        starts[slot] = i;
        seg_lo[slot] = s0;
        seg_hi[slot] = s1;
      }
      __syncwarp();
      if (threadIdx.x == 0) nstart += __popc(ball);
      __syncwarp();
    }
  }
  __syncthreads();
  const int C4 = C / 4, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int p = warp; p < nstart; p += nwarps) {  // one warp per piece
    const int i = starts[p], s0 = seg_lo[p], s1 = seg_hi[p];
    const int end = min(s1, i + ENC_PIECE);
    const uint32_t id = sorted[i] / (uint32_t)M;
    // lane l holds the 16-byte columns l, l + 32, ... (C <= 1024: at most 8);
    // a row's loads are all issued before its additions, rows in order
    float4 s[8];
#pragma unroll
    for (int k = 0; k < 8; k++) s[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int j = i; j < end; j++) {
      const float4* row = reinterpret_cast<const float4*>(dout + (int64_t)(sorted[j] % (uint32_t)M) * C);
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; k++) v[k] = lane + 32 * k < C4 ? __ldg(row + lane + 32 * k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; k++) { s[k].x += v[k].x; s[k].y += v[k].y; s[k].z += v[k].z; s[k].w += v[k].w; }
    }
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const int c4 = lane + 32 * k;
      if (c4 >= C4) break;
      if (s1 - s0 <= ENC_PIECE) {
        float4* d = reinterpret_cast<float4*>(dwte + (int64_t)id * C) + c4;
        float4 o = *d;
        o.x += s[k].x; o.y += s[k].y; o.z += s[k].z; o.w += s[k].w;
        *d = o;
      } else {
        reinterpret_cast<float4*>(partial + (int64_t)i * C)[c4] = s[k];
      }
    }
  }
}

// Block b: the segments that start in [64b, 64b+64) and have more than one
// piece add their pieces' partials in order into dwte.
__global__ void encoder_bwd_combine_kernel(float* dwte, const float* partial,
                                           const uint32_t* sorted, int M, int C) {
  pdl_trigger();
  pdl_wait();
  __shared__ int starts[ENC_RANGE], ends[ENC_RANGE];
  __shared__ int nstart;
  const int i0 = blockIdx.x * ENC_RANGE;
  if (threadIdx.x == 0) nstart = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    for (int k = threadIdx.x; k < ENC_RANGE; k += 32) {
      const int i = i0 + k;
      bool take = false;
      int s1 = 0;
      if (i < M) {
        const uint32_t id = sorted[i] / (uint32_t)M;
        if (i == 0 || sorted[i - 1] / (uint32_t)M != id) {
          s1 = lower_bound_u32(sorted, M, (id + 1) * (uint32_t)M);
          take = s1 - i > ENC_PIECE;
        }
      }
      const uint32_t ball = __ballot_sync(0xffffffffu, take);
      const int slot = nstart + __popc(ball & ((1u << threadIdx.x) - 1u));
      if (take) {
        starts[slot] = i;
        ends[slot] = s1;
      }
      __syncwarp();
      if (threadIdx.x == 0) nstart += __popc(ball);
      __syncwarp();
    }
  }
  __syncthreads();
  const int C4 = C / 4, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int p = warp; p < nstart; p += nwarps) {  // one warp per segment
    const int i = starts[p], s1 = ends[p];
    const uint32_t id = sorted[i] / (uint32_t)M;
    float4 s[8];
#pragma unroll
    for (int k = 0; k < 8; k++) s[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = i; j < s1; j += ENC_PIECE) {  // the pieces' partials, in order
      const float4* row = reinterpret_cast<const float4*>(partial + (int64_t)j * C);
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; k++) v[k] = lane + 32 * k < C4 ? row[lane + 32 * k] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; k++) { s[k].x += v[k].x; s[k].y += v[k].y; s[k].z += v[k].z; s[k].w += v[k].w; }
    }
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const int c4 = lane + 32 * k;
      if (c4 >= C4) break;
      float4* d = reinterpret_cast<float4*>(dwte + (int64_t)id * C) + c4;
      float4 o = *d;
      o.x += s[k].x; o.y += s[k].y; o.z += s[k].z; o.w += s[k].w;
      *d = o;
    }
  }
}

void launch_encoder_bwd(LaunchCtx& c, float* dwte, float* dwpe, const float* dout,
                        const int32_t* tok, int B, int T, int C, int Vp, uint32_t* sorted,
                        float* partial) {
  const int M = B * T;
  {
    const int64_t n = (int64_t)T * C;
    int grid = (int)std::min<int64_t>(cdiv(n, 256), (int64_t)c.num_sms * 8);
    launch_pdl(c, encoder_bwd_wpe_kernel, dim3(grid), dim3(256), 0, dwpe, dout, B, T, C);
  }
  // the sort's second key buffer borrows the head of the piece partials,
  // which are written only after the sort
  const size_t smem = (size_t)ES_BINS * ES_WARPS * sizeof(int);
  cudaFuncSetAttribute(encoder_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(c, encoder_sort_kernel, dim3(1), dim3(ES_THREADS), smem, sorted, reinterpret_cast<uint32_t*>(partial),
             tok, M, Vp);
  launch_pdl(c, encoder_bwd_piece_kernel, dim3(cdiv(M, ENC_RANGE)), dim3(256), 0, dwte, partial, dout, sorted, M, C);
  launch_pdl(c, encoder_bwd_combine_kernel, dim3(cdiv(M, ENC_RANGE)), dim3(256), 0, dwte, partial, sorted, M, C);
}

// 8 values at p (16-byte aligned for bf16, 32 for float), one or two 16-byte stores
template <typename OutT>
__device__ __forceinline__ void store8(OutT* p, const float* v);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<bf16>(bf16* p, const float* v) {
  uint4 u;
  __nv_bfloat162 t = __floats2bfloat162_rn(v[0], v[1]);
  u.x = *reinterpret_cast<uint32_t*>(&t);
  t = __floats2bfloat162_rn(v[2], v[3]);
  u.y = *reinterpret_cast<uint32_t*>(&t);
  t = __floats2bfloat162_rn(v[4], v[5]);
  u.z = *reinterpret_cast<uint32_t*>(&t);
  t = __floats2bfloat162_rn(v[6], v[7]);
  u.w = *reinterpret_cast<uint32_t*>(&t);
  *reinterpret_cast<uint4*>(p) = u;
}

// ============================================================ LayerNorm
template <typename OutT>
__device__ __forceinline__ void store4(OutT* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<bf16>(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
  return make_float4(a.x, a.y, b.x, b.y);
}

// One warp per row: mean, then variance about the mean (two passes; the row
// stays in L1), then y = (x - mean) * rstd * w + b.
// One warp per row, rows strided over a grid of ~2 blocks per SM.  Lane l
// holds the float4 column chunks l, l+32, ... (NCH = ceil(C/128)) of the
// row in registers, so the row is read from HBM once; the next row's loads
// are issued before this row is reduced.  mean = sum/C, var = sum((x -
// mean)^2)/C (two passes over the registers), rstd = 1/sqrt(var + 1e-5).
template <typename OutT, int NCH>
__global__ void __launch_bounds__(256) layernorm_fwd_kernel(OutT* out, float* mean, float* rstd,
                                                            const float* inp, const float* w,
                                                            const float* b, int N, int C) {
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  float4 wv[NCH], bv[NCH], xv[NCH];
#pragma unroll
  for (int k = 0; k < NCH; k++) {
    const int c = (lane + 32 * k) * 4;
    wv[k] = bv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < C) {
      wv[k] = *reinterpret_cast<const float4*>(w + c);
      bv[k] = *reinterpret_cast<const float4*>(b + c);
    }
  }
  pdl_wait();
  int row = blockIdx.x * (blockDim.x >> 5) + warp;
#pragma unroll
  for (int k = 0; k < NCH; k++) {
    const int c = (lane + 32 * k) * 4;
    xv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < N && c < C) xv[k] = *reinterpret_cast<const float4*>(inp + (int64_t)row * C + c);
  }
  for (; row < N; row += nwarps) {
    float4 nx[NCH];
    const int nrow = row + nwarps;
#pragma unroll
    for (int k = 0; k < NCH; k++) {
      const int c = (lane + 32 * k) * 4;
      nx[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (nrow < N && c < C) nx[k] = *reinterpret_cast<const float4*>(inp + (int64_t)nrow * C + c);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NCH; k++) s += (xv[k].x + xv[k].y) + (xv[k].z + xv[k].w);
    const float m = warp_sum(s) / (float)C;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < NCH; k++) {
      if ((lane + 32 * k) * 4 < C) {
        const float a = xv[k].x - m, bb = xv[k].y - m, cc = xv[k].z - m, d = xv[k].w - m;
        q += (a * a + bb * bb) + (cc * cc + d * d);
      }
    }
    const float var = warp_sum(q) / (float)C;
    const float r = 1.f / sqrtf(var + 1e-5f);
    OutT* y = out + (int64_t)row * C;
#pragma unroll
    for (int k = 0; k < NCH; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C)
        store4<OutT>(y + c, (xv[k].x - m) * r * wv[k].x + bv[k].x, (xv[k].y - m) * r * wv[k].y + bv[k].y,
                     (xv[k].z - m) * r * wv[k].z + bv[k].z, (xv[k].w - m) * r * wv[k].w + bv[k].w);
    }
    if (lane == 0) { mean[row] = m; rstd[row] = r; }
#pragma unroll
    for (int k = 0; k < NCH; k++) xv[k] = nx[k];
  }
}

template <typename OutT, int NCH>
static void ln_fwd_launch(LaunchCtx& c, OutT* out, float* mean, float* rstd, const float* inp,
                          const float* w, const float* b, int N, int C) {
  const int blocks = std::min(cdiv(N, 8), 2 * c.num_sms);
  launch_pdl(c, layernorm_fwd_kernel<OutT, NCH>, dim3(blocks), dim3(256), 0, out, mean, rstd, inp, w, b, N, C);
}

template <typename OutT>
void launch_layernorm_fwd(LaunchCtx& c, OutT* out, float* mean, float* rstd, const float* inp,
                          const float* w, const float* b, int N, int C) {
  switch ((C + 127) / 128) {  // C <= 1024
    case 1: ln_fwd_launch<OutT, 1>(c, out, mean, rstd, inp, w, b, N, C); break;
    case 2: ln_fwd_launch<OutT, 2>(c, out, mean, rstd, inp, w, b, N, C); break;
    case 3: ln_fwd_launch<OutT, 3>(c, out, mean, rstd, inp, w, b, N, C); break;
    case 4: ln_fwd_launch<OutT, 4>(c, out, mean, rstd, inp, w, b, N, C); break;
    case 5: ln_fwd_launch<OutT, 5>(c, out, mean, rstd, inp, w, b, N, C); break;
    case 6: ln_fwd_launch<OutT, 6>(c, out, mean, rstd, inp, w, b, N, C); break;
    case 7: ln_fwd_launch<OutT, 7>(c, out, mean, rstd, inp, w, b, N, C); break;
    default: ln_fwd_launch<OutT, 8>(c, out, mean, rstd, inp, w, b, N, C); break;
  }
}
template void launch_layernorm_fwd<float>(LaunchCtx&, float*, float*, float*, const float*,
                                          const float*, const float*, int, int);
template void launch_layernorm_fwd<bf16>(LaunchCtx&, bf16*, float*, float*, const float*,
                                         const float*, const float*, int, int);

#define LNB_WARPS 8
#define LNB_STAGES 2        // rows in flight per warp
#define LNB_ROWS_PER_BLOCK 64  // rows per block at least (grid sizing)

// partial rows: one per block of a grid of at most cdiv(N, 64) blocks
int64_t ln_partial_floats(int N, int C) { return (int64_t)cdiv(N, LNB_ROWS_PER_BLOCK) * 3 * C; }

static size_t lnb_smem(int C) {
  return (size_t)LNB_WARPS * LNB_STAGES * 3 * C * sizeof(float) + LNB_WARPS * LNB_STAGES * sizeof(uint64_t);
}

// One warp per row, rows strided over a persistent grid.  Each warp streams
// its rows (dy, x and, when accumulating, the old residual gradient) into
// its own LNB_STAGES-deep shared-memory ring with bulk copies, so the next
// rows' loads are in flight while this one is processed from shared memory.
// Lane l owns the float4 column chunks l, l+32, ... (NCH = C/128 of them)
// and keeps its gamma / beta / residual-gradient column partials in
// registers across all of the warp's rows; the block adds its warps'
// partials in warp order into one partial row, and reduce_partials_kernel
// adds the blocks' rows in order.
//   xhat = (x - mean) rstd, g = dy * gamma,
//   dx = rstd (g - mean(g) - xhat mean(g xhat)),  dres (+)= dx.
// Four consecutive values as fp32 (a 16-byte fp32 or an 8-byte bf16 load).
__device__ __forceinline__ float4 load4f(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4f(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename ActT, int NCH>
__global__ void __launch_bounds__(LNB_WARPS * 32, 1)
    layernorm_bwd_kernel(float* dres, ActT* dres_act, float* partial, const ActT* dy,
                         const float* inp, const float* w, const float* mean, const float* rstd,
                         int N, int C, int accumulate, int* err) {
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t lnb_sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* ring = reinterpret_cast<float*>(lnb_sm) + (size_t)warp * LNB_STAGES * 3 * C;
  uint64_t* bars = reinterpret_cast<uint64_t*>(lnb_sm + (size_t)LNB_WARPS * LNB_STAGES * 3 * C * sizeof(float)) +
                   warp * LNB_STAGES;
  if (lane == 0) {
    for (int s = 0; s < LNB_STAGES; s++) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  float4 wv[NCH], pw[NCH], pb[NCH], pr[NCH];
#pragma unroll
  for (int k = 0; k < NCH; k++) {
    const int c = (lane + 32 * k) * 4;
    pw[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    pb[k] = pw[k];
    pr[k] = pw[k];
    wv[k] = pw[k];
    if (c < C) wv[k] = *reinterpret_cast<const float4*>(w + c);
  }
  pdl_wait();  // from here on global memory written by the previous kernel is read
  const int gw = blockIdx.x * LNB_WARPS + warp, nw = gridDim.x * LNB_WARPS;
  const uint32_t rowbytes = (uint32_t)C * sizeof(float), dybytes = (uint32_t)C * sizeof(ActT);
  auto issue = [&](int row, int s) {
    float* st = ring + (size_t)s * 3 * C;  // dy (C values of ActT) | x | old dres
    mbar_arrive_expect_tx(&bars[s], (accumulate ? 2u : 1u) * rowbytes + dybytes);
    bulk_load(st, dy + (int64_t)row * C, dybytes, &bars[s]);
    bulk_load(st + C, inp + (int64_t)row * C, rowbytes, &bars[s]);
    if (accumulate) bulk_load(st + 2 * C, dres + (int64_t)row * C, rowbytes, &bars[s]);
  };
  if (lane == 0)
    for (int s = 0; s < LNB_STAGES; s++)
      if (gw + s * nw < N) issue(gw + s * nw, s);
  float m = 0.f, r = 0.f;
  if (gw < N) { m = mean[gw]; r = rstd[gw]; }
  int it = 0;
  for (int row = gw; row < N; row += nw, it++) {
    const int s = it % LNB_STAGES;
    const int nrow = row + nw;
    float mn = 0.f, rn = 0.f;  // next row's statistics, loaded ahead
    if (nrow < N) { mn = mean[nrow]; rn = rstd[nrow]; }
    mbar_wait(&bars[s], (uint32_t)(it / LNB_STAGES) & 1u, err);
    const ActT* g = reinterpret_cast<const ActT*>(ring + (size_t)s * 3 * C);
    const float* x = ring + (size_t)s * 3 * C + C;
    const float* o = x + C;
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int k = 0; k < NCH; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        const float4 xv = *reinterpret_cast<const float4*>(x + c);
        const float4 gv = load4f(g + c);
        const float h0 = gv.x * wv[k].x, h1 = gv.y * wv[k].y, h2 = gv.z * wv[k].z, h3 = gv.w * wv[k].w;
        s1 += (h0 + h1) + (h2 + h3);
        s2 += (h0 * (xv.x - m) * r + h1 * (xv.y - m) * r) + (h2 * (xv.z - m) * r + h3 * (xv.w - m) * r);
      }
    }
    const float mg = warp_sum(s1) / (float)C;
    const float mgx = warp_sum(s2) / (float)C;
    float* dr = dres + (int64_t)row * C;
#pragma unroll
    for (int k = 0; k < NCH; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        const float4 xv = *reinterpret_cast<const float4*>(x + c);
        const float4 gv = load4f(g + c);
        const float x0 = (xv.x - m) * r, x1 = (xv.y - m) * r, x2 = (xv.z - m) * r, x3 = (xv.w - m) * r;
        float4 d;
        d.x = r * (gv.x * wv[k].x - mg - x0 * mgx);
        d.y = r * (gv.y * wv[k].y - mg - x1 * mgx);
        d.z = r * (gv.z * wv[k].z - mg - x2 * mgx);
        d.w = r * (gv.w * wv[k].w - mg - x3 * mgx);
        if (accumulate) {
          const float4 ov = *reinterpret_cast<const float4*>(o + c);
          d.x += ov.x; d.y += ov.y; d.z += ov.z; d.w += ov.w;
        }
        *reinterpret_cast<float4*>(dr + c) = d;
        if (dres_act) store4<ActT>(dres_act + (int64_t)row * C + c, d.x, d.y, d.z, d.w);
        pw[k].x += gv.x * x0; pw[k].y += gv.y * x1; pw[k].z += gv.z * x2; pw[k].w += gv.w * x3;
        pb[k].x += gv.x; pb[k].y += gv.y; pb[k].z += gv.z; pb[k].w += gv.w;
        pr[k].x += d.x; pr[k].y += d.y; pr[k].z += d.z; pr[k].w += d.w;
      }
    }
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && row + LNB_STAGES * nw < N) issue(row + LNB_STAGES * nw, s);
    m = mn;
    r = rn;
  }
  // the block's partial row: each warp leaves its column partials in its own
  // (now idle) ring area, then the block adds the 8 warps' rows in warp
  // order (a fixed order) and writes one row of 3C
  float* mine = ring;
#pragma unroll
  for (int k = 0; k < NCH; k++) {
    const int c = (lane + 32 * k) * 4;
    if (c < C) {
      *reinterpret_cast<float4*>(mine + c) = pw[k];
      *reinterpret_cast<float4*>(mine + C + c) = pb[k];
      *reinterpret_cast<float4*>(mine + 2 * C + c) = pr[k];
    }
  }
  __syncthreads();
  const float* rings = reinterpret_cast<const float*>(lnb_sm);
  float* out = partial + (int64_t)blockIdx.x * 3 * C;
  for (int c = threadIdx.x * 4; c < 3 * C; c += LNB_WARPS * 32 * 4) {
    float4 t = *reinterpret_cast<const float4*>(rings + c);
#pragma unroll
    for (int w2 = 1; w2 < LNB_WARPS; w2++) {
      const float4 u = *reinterpret_cast<const float4*>(rings + (size_t)w2 * LNB_STAGES * 3 * C + c);
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    *reinterpret_cast<float4*>(out + c) = t;
  }
}

// Sum nb partial rows of width W = parts * seg and add segment i into
// d[i][0:seg] (a null d[i] is skipped).  Block: 32 columns x 32 row groups;
// group g sums rows g, g+32, ... in order, then the 32 group sums are added
// in group order (a fixed order: the result repeats bit for bit).
#define RP_COLS 32
#define RP_GROUPS 32
__global__ void __launch_bounds__(RP_COLS * RP_GROUPS)
    reduce_partials_kernel(float* d0, float* d1, float* d2, const float* partial, int nb, int W, int seg) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm[RP_GROUPS][RP_COLS + 1];
  const int lane = threadIdx.x % RP_COLS, grp = threadIdx.x / RP_COLS;
  const int c = blockIdx.x * RP_COLS + lane;
  float s = 0.f;
  if (c < W) {
#pragma unroll 4
    for (int b = grp; b < nb; b += RP_GROUPS) s += partial[(int64_t)b * W + c];
  }
  sm[grp][lane] = s;
  __syncthreads();
  if (grp == 0 && c < W) {
    float* d = c < seg ? d0 : (c < 2 * seg ? d1 : d2);
    if (!d) return;
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < RP_GROUPS; q++) t += sm[q][lane];
    d[c % seg] += t;
  }
}

// reduce_partials_kernel over a list of jobs: block b works on the job with
// the largest first_block <= b, on its column block b - first_block.  Many
// small reductions in one launch keep more loads in flight than one launch
// each, and take one step of the stream's dependency chain instead of one
// per reduction.
__global__ void __launch_bounds__(RP_COLS * RP_GROUPS) reduce_jobs_kernel(const ReduceJob* jobs, int njobs) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm[RP_GROUPS][RP_COLS + 1];
  __shared__ int sj;
  if (threadIdx.x == 0) {
    int lo = 0, hi = njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (jobs[mid].first_block <= (int)blockIdx.x) lo = mid;
      else hi = mid - 1;
    }
    sj = lo;
  }
  __syncthreads();
  const ReduceJob& jb = jobs[sj];
  const int lane = threadIdx.x % RP_COLS, grp = threadIdx.x / RP_COLS;
  const int W = jb.W, nb = jb.nb, seg = jb.seg;
  const int c = ((int)blockIdx.x - jb.first_block) * RP_COLS + lane;
  const float* partial = jb.partial;
  float s = 0.f;
  if (c < W) {
#pragma unroll 4
    for (int b = grp; b < nb; b += RP_GROUPS) s += partial[(int64_t)b * W + c];
  }
  sm[grp][lane] = s;
  __syncthreads();
  if (grp == 0 && c < W) {
    float* d = c < seg ? jb.d[0] : (c < 2 * seg ? jb.d[1] : jb.d[2]);
    if (!d) return;
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < RP_GROUPS; q++) t += sm[q][lane];
    d[c % seg] += t;
  }
}

int reduce_job_blocks(int W) { return cdiv(W, RP_COLS); }

void launch_reduce_jobs(LaunchCtx& c, const ReduceJob* jobs, int njobs, int blocks) {
  if (njobs <= 0 || blocks <= 0) return;
  launch_pdl(c, reduce_jobs_kernel, dim3(blocks), dim3(RP_COLS * RP_GROUPS), 0, jobs, njobs);
}

template <typename ActT, int NCH>
static void ln_bwd_launch(LaunchCtx& c, int nb, float* dres, ActT* dres_act, float* partial,
                          const ActT* dy, const float* inp, const float* w, const float* mean,
                          const float* rstd, int N, int C, bool accumulate) {
  const size_t smem = lnb_smem(C);
  cudaFuncSetAttribute(layernorm_bwd_kernel<ActT, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  launch_pdl(c, layernorm_bwd_kernel<ActT, NCH>, dim3(nb), dim3(LNB_WARPS * 32), smem, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate ? 1 : 0, c.err);
}

template <typename ActT>
int launch_layernorm_bwd_partials(LaunchCtx& c, float* dres, ActT* dres_act, const ActT* dy, const float* inp,
                                  const float* w, const float* mean, const float* rstd, int N, int C,
                                  bool accumulate, float* partial) {
  int nb = cdiv(N, LNB_ROWS_PER_BLOCK);  // one partial row per block: nb <= ln_partial_floats / (3C)
  if (c.num_sms > 0) nb = std::min(nb, c.num_sms);
  switch ((C + 127) / 128) {  // C <= 1024 (checked by the callers): partials in registers
    case 1: ln_bwd_launch<ActT, 1>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    case 2: ln_bwd_launch<ActT, 2>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    case 3: ln_bwd_launch<ActT, 3>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    case 4: ln_bwd_launch<ActT, 4>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    case 5: ln_bwd_launch<ActT, 5>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    case 6: ln_bwd_launch<ActT, 6>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    case 7: ln_bwd_launch<ActT, 7>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
    default: ln_bwd_launch<ActT, 8>(c, nb, dres, dres_act, partial, dy, inp, w, mean, rstd, N, C, accumulate); break;
  }
  return nb;
}
template int launch_layernorm_bwd_partials<float>(LaunchCtx&, float*, float*, const float*, const float*,
                                                  const float*, const float*, const float*, int, int, bool,
                                                  float*);
template int launch_layernorm_bwd_partials<bf16>(LaunchCtx&, float*, bf16*, const bf16*, const float*,
                                                 const float*, const float*, const float*, int, int, bool,
                                                 float*);

template <typename ActT>
void launch_layernorm_bwd(LaunchCtx& c, float* dres, ActT* dres_act, float* dw, float* db,
                          float* dres_colsum, const ActT* dy, const float* inp, const float* w,
                          const float* mean, const float* rstd, int N, int C, bool accumulate,
                          float* partial) {
  const int nb = launch_layernorm_bwd_partials<ActT>(c, dres, dres_act, dy, inp, w, mean, rstd, N, C, accumulate,
                                                     partial);
  launch_pdl(c, reduce_partials_kernel, dim3(cdiv(3 * C, RP_COLS)), dim3(RP_COLS * RP_GROUPS), 0, dw, db, dres_colsum, partial, nb, 3 * C, C);
}
template void launch_layernorm_bwd<float>(LaunchCtx&, float*, float*, float*, float*, float*,
                                          const float*, const float*, const float*, const float*,
                                          const float*, int, int, bool, float*);
template void launch_layernorm_bwd<bf16>(LaunchCtx&, float*, bf16*, float*, float*, float*,
                                         const bf16*, const float*, const float*, const float*,
                                         const float*, int, int, bool, float*);

// ============================================================ column sums
#define CS_CHUNKS 128
int64_t colsum_partial_floats(int M, int N) { return (int64_t)CS_CHUNKS * N; }

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<bf16>(const bf16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// grid (ceil(N/256), CS_CHUNKS), 256 threads: 8 row groups x 32 threads x 8
// columns (16-byte loads for bf16).  Group g sums rows r0+g, r0+g+8, ... of
// the chunk in order; the 8 group sums are added in group order.
template <typename T>
__global__ void __launch_bounds__(256) colsum_partial_kernel(float* partial, const T* x, int M, int N, int64_t ld) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sg[8][256];
  const int grp = threadIdx.x >> 5, t = threadIdx.x & 31;
  const int col = blockIdx.x * 256 + t * 8;
  const int rows = (M + CS_CHUNKS - 1) / CS_CHUNKS;
  const int r0 = blockIdx.y * rows, r1 = min(M, r0 + rows);
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (col < N) {
#pragma unroll 4
    for (int r = r0 + grp; r < r1; r += 8) {
      float v[8];
      load8<T>(x + (int64_t)r * ld + col, v);
#pragma unroll
      for (int j = 0; j < 8; j++) s[j] += v[j];
    }
  }
#pragma unroll
  for (int j = 0; j < 8; j++) sg[grp][t * 8 + j] = s[j];
  __syncthreads();
  const int cc = threadIdx.x;  // one column of the block each
  if (blockIdx.x * 256 + cc < N) {
    float o = 0.f;
#pragma unroll
    for (int q = 0; q < 8; q++) o += sg[q][cc];
    partial[(int64_t)blockIdx.y * N + blockIdx.x * 256 + cc] = o;
  }
}

template <typename T>
int launch_colsum_partials(LaunchCtx& c, float* partial, const T* x, int M, int N, int64_t ld) {
  dim3 grid(cdiv(N, 256), CS_CHUNKS);
  launch_pdl(c, colsum_partial_kernel<T>, dim3(grid), dim3(256), 0, partial, x, M, N, ld);
  return CS_CHUNKS;
}
template int launch_colsum_partials<float>(LaunchCtx&, float*, const float*, int, int, int64_t);
template int launch_colsum_partials<bf16>(LaunchCtx&, float*, const bf16*, int, int, int64_t);



// ============================================================ softmax + cross-entropy
#define LOG2E 1.4426950408889634f

// (m, s) pairs: a running maximum m (natural units) and s = sum of e^(x - m).
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) return;
  s = s * ex2_hw((m - mm) * LOG2E) + s2 * ex2_hw((m2 - mm) * LOG2E);
  m = mm;
}

// One block per row.  Pass 1 reads 8 logits at a time and folds each group
// into the running (max, sum of e^(x - max)) -- one max and one rescale per
// group of 8, each e^(x - m) one FFMA and one ex2 -- then a block reduction
// gives lse.  Pass 2 (the row is now in L2) writes
//   dlogits = (e^(x - lse) - onehot(target)) * dscale,  pad columns 0,
// in place; only the group holding the target and the groups past V take
// the slow path.  loss = lse - logit[target].
template <typename T>
__global__ void __launch_bounds__(512) crossentropy_kernel(T* logits, float* losses, const int32_t* targets, int V,
                                    int Vp, float dscale, int write_dlogits, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm_m[32], sm_s[32];
  const int64_t row = blockIdx.x;
  T* l = logits + row * Vp;
  int tg = targets ? targets[row] : -1;
  if (targets && (tg < 0 || tg >= V)) {
    if (threadIdx.x == 0) record_error(err, DEVERR_TOKEN);
    tg = 0;
  }
  const float lt = targets ? to_f(l[tg]) : 0.f;  // read before any thread overwrites the row
  float m = -INFINITY, s = 0.f;
  const int nch = Vp / 8;
  for (int q = threadIdx.x; q < nch; q += blockDim.x) {
    float v[8];
    load8<T>(l + q * 8, v);
    const int base = q * 8;
    if (base + 8 > V) {
#pragma unroll
      for (int j = 0; j < 8; j++) v[j] = base + j < V ? v[j] : -INFINITY;
    }
    float cm = v[0];
#pragma unroll
    for (int j = 1; j < 8; j++) cm = fmaxf(cm, v[j]);
    if (cm == -INFINITY) continue;
    const float nm = fmaxf(m, cm), nl = -nm * LOG2E;
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) a += ex2_hw(fmaf(v[j], LOG2E, nl));
    s = s * ex2_hw((m - nm) * LOG2E) + a;
    m = nm;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (lane == 0) { sm_m[warp] = m; sm_s[warp] = s; }
  __syncthreads();
  if (warp == 0) {
    m = lane < nw ? sm_m[lane] : -INFINITY;
    s = lane < nw ? sm_s[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_combine(m, s, m2, s2);
    }
    if (lane == 0) { sm_m[0] = m; sm_s[0] = s; }
  }
  __syncthreads();
  const float lse = sm_m[0] + logf(sm_s[0]);
  if (threadIdx.x == 0 && targets) losses[row] = lse - lt;
  if (!write_dlogits) return;
  const float nl = -lse * LOG2E;
  for (int q = threadIdx.x; q < nch; q += blockDim.x) {
    float v[8];
    load8<T>(l + q * 8, v);
    const int base = q * 8;
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; j++) o[j] = ex2_hw(fmaf(v[j], LOG2E, nl)) * dscale;
    if (base + 8 > V || (base <= tg && tg < base + 8)) {
#pragma unroll
      for (int j = 0; j < 8; j++) {
        if (base + j >= V) o[j] = 0.f;
        else if (base + j == tg) o[j] -= dscale;
      }
    }
    store4<T>(l + base, o[0], o[1], o[2], o[3]);
    store4<T>(l + base + 4, o[4], o[5], o[6], o[7]);
  }
}

// The same computation with the row staged in shared memory: one thread
// starts bulk copies of the whole row (pieces of CE_PIECE bytes, each on
// its own mbarrier) before any arithmetic, so that a block keeps the full
// row in flight; pass 1 folds each group of 8 into (max, sum) once its
// piece has landed, pass 2 reads the row from shared memory and writes
// dlogits with coalesced 16-byte stores.  The row is read from HBM once.
#define CE_PIECE 16384
#define CE_MAX_PIECES 14
template <typename T>
__global__ void __launch_bounds__(512) crossentropy_smem_kernel(T* logits, float* losses, const int32_t* targets,
                                                                 int V, int Vp, float dscale, int write_dlogits,
                                                                 int* err) {
  extern __shared__ __align__(128) uint8_t ce_row[];
  __shared__ uint64_t bar[CE_MAX_PIECES];
  __shared__ float sm_m[32], sm_s[32];
  const int64_t row = blockIdx.x;
  T* l = logits + row * Vp;
  const T* r = reinterpret_cast<const T*>(ce_row);
  const uint32_t rowbytes = (uint32_t)Vp * sizeof(T);
  const int np = (int)((rowbytes + CE_PIECE - 1) / CE_PIECE);
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int q = 0; q < np; q++) mbar_init(&bar[q], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int q = 0; q < np; q++) {
      const uint32_t b = min((uint32_t)CE_PIECE, rowbytes - (uint32_t)q * CE_PIECE);
      mbar_arrive_expect_tx(&bar[q], b);
      bulk_load(ce_row + (size_t)q * CE_PIECE, reinterpret_cast<const uint8_t*>(l) + (size_t)q * CE_PIECE, b, &bar[q]);
    }
  }
  int tg = targets ? targets[row] : -1;
  if (targets && (tg < 0 || tg >= V)) {
    if (threadIdx.x == 0) record_error(err, DEVERR_TOKEN);
    tg = 0;
  }
  constexpr int GB = 8 * sizeof(T);  // bytes of a group of 8
  int landed = 0;                     // pieces this thread has seen complete
  float m = -INFINITY, s = 0.f;
  const int nch = Vp / 8;
  for (int q = threadIdx.x; q < nch; q += blockDim.x) {
    const int pc = q * GB / CE_PIECE;
    while (landed <= pc) mbar_wait(&bar[landed++], 0u, err);
    float v[8];
    load8<T>(r + q * 8, v);
    const int base = q * 8;
    if (base + 8 > V) {
#pragma unroll
      for (int j = 0; j < 8; j++) v[j] = base + j < V ? v[j] : -INFINITY;
    }
    float cm = v[0];
#pragma unroll
    for (int j = 1; j < 8; j++) cm = fmaxf(cm, v[j]);
    if (cm == -INFINITY) continue;
    const float nm = fmaxf(m, cm), nl = -nm * LOG2E;
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) a += ex2_hw(fmaf(v[j], LOG2E, nl));
    s = s * ex2_hw((m - nm) * LOG2E) + a;
    m = nm;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (lane == 0) { sm_m[warp] = m; sm_s[warp] = s; }
  __syncthreads();
  if (warp == 0) {
    m = lane < nw ? sm_m[lane] : -INFINITY;
    s = lane < nw ? sm_s[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_combine(m, s, m2, s2);
    }
    if (lane == 0) { sm_m[0] = m; sm_s[0] = s; }
  }
  __syncthreads();
  const float lse = sm_m[0] + logf(sm_s[0]);
  if (threadIdx.x == 0 && targets) {
    const int pc = tg * (int)sizeof(T) / CE_PIECE;
    while (landed <= pc) mbar_wait(&bar[landed++], 0u, err);
    losses[row] = lse - to_f(r[tg]);
  }
  if (!write_dlogits) return;
  const float nl = -lse * LOG2E;
  for (int q = threadIdx.x; q < nch; q += blockDim.x) {
    const int pc = q * GB / CE_PIECE;
    while (landed <= pc) mbar_wait(&bar[landed++], 0u, err);
    float v[8];
    load8<T>(r + q * 8, v);
    const int base = q * 8;
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; j++) o[j] = ex2_hw(fmaf(v[j], LOG2E, nl)) * dscale;
    if (base + 8 > V || (base <= tg && tg < base + 8)) {
#pragma unroll
      for (int j = 0; j < 8; j++) {
        if (base + j >= V) o[j] = 0.f;
        else if (base + j == tg) o[j] -= dscale;
      }
    }
    store8<T>(l + base, o);
  }
}

template <typename T>
void launch_crossentropy(LaunchCtx& c, T* logits, float* losses, const int32_t* targets, int M,
                         int V, int Vp, float dscale, bool dlogits) {
  const size_t rowbytes = (size_t)Vp * sizeof(T);
  if (rowbytes <= (size_t)CE_PIECE * CE_MAX_PIECES && rowbytes % 16 == 0 &&
      reinterpret_cast<uintptr_t>(logits) % 16 == 0) {
    static bool attr = false;
    if (!attr) {
      cudaFuncSetAttribute(crossentropy_smem_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CE_PIECE * CE_MAX_PIECES);
      attr = true;
    }
    launch_pdl(c, crossentropy_smem_kernel<T>, dim3(M), dim3(512), rowbytes, logits, losses, targets, V, Vp,
               dscale, dlogits ? 1 : 0, c.err);
    return;
  }
  launch_pdl(c, crossentropy_kernel<T>, dim3(M), dim3(512), 0, logits, losses, targets, V, Vp, dscale,
                                                  dlogits ? 1 : 0, c.err);
}
template void launch_crossentropy<float>(LaunchCtx&, float*, float*, const int32_t*, int, int, int,
                                         float, bool);
template void launch_crossentropy<bf16>(LaunchCtx&, bf16*, float*, const int32_t*, int, int, int,
                                        float, bool);

__global__ void mean_kernel(float* out, const float* x, int M) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < M; i += blockDim.x) s += x[i];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < (blockDim.x >> 5) ? sm[threadIdx.x] : 0.f;
    s = warp_sum(s);
    if (threadIdx.x == 0) out[0] = s / (float)M;
  }
}
void launch_mean(LaunchCtx& c, float* out, const float* losses, int M) {
  launch_pdl(c, mean_kernel, dim3(1), dim3(1024), 0, out, losses, M);
}

// ============================================================ AdamW
__global__ void adamw_kernel(float* p, const float* g, float* m, float* v, bf16* shadow, int64_t n4,
                             float lr, float b1, float b2, float eps, float wd, float c1,
                             float c2) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 pp = reinterpret_cast<float4*>(p)[i];
    const float4 gg = reinterpret_cast<const float4*>(g)[i];
    float4 mm = reinterpret_cast<float4*>(m)[i];
    float4 vv = reinterpret_cast<float4*>(v)[i];
    float* P = &pp.x;
    const float* G = &gg.x;
    float* Mm = &mm.x;
    float* Vv = &vv.x;
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const float mi = b1 * Mm[q] + (1.f - b1) * G[q];
      const float vi = b2 * Vv[q] + (1.f - b2) * G[q] * G[q];
      Mm[q] = mi;
      Vv[q] = vi;
      const float mh = mi / c1, vh = vi / c2;
      P[q] = P[q] - lr * (mh / (sqrtf(vh) + eps) + wd * P[q]);
    }
    reinterpret_cast<float4*>(p)[i] = pp;
    reinterpret_cast<float4*>(m)[i] = mm;
    reinterpret_cast<float4*>(v)[i] = vv;
    if (shadow) store4<bf16>(shadow + i * 4, pp.x, pp.y, pp.z, pp.w);
  }
}

void launch_adamw(LaunchCtx& c, float* p, const float* g, float* m, float* v, bf16* shadow,
                  int64_t n, float lr, float b1, float b2, float eps, float wd, float c1,
                  float c2) {
  const int64_t n4 = n / 4;  // the parameter count is a multiple of 4 (C % 8 == 0)
  int grid = (int)std::min<int64_t>(cdiv(n4, 256), (int64_t)c.num_sms * 16);
  launch_pdl(c, adamw_kernel, dim3(grid), dim3(256), 0, p, g, m, v, shadow, n4, lr, b1, b2, eps, wd, c1, c2);
}

// ============================================================ allocation-free LayerNorm backward
// gpt2_layernorm_backward_noalloc: the LayerNorm backward above for callers
// that cannot allocate device memory.  Its partial sums (at most
// ceil(N/64) rows of 3*C floats) live in this file-scope array instead of caller- or
// model-owned scratch; every GPU that loads the library holds it until the
// process exits.  Its bounded waits report into g_noalloc_err, which
// gpt2_noalloc_check reads and clears.
#define NOALLOC_SCRATCH_FLOATS (1 << 21)  // 8 MiB
static __device__ __align__(256) float g_noalloc_scratch[NOALLOC_SCRATCH_FLOATS];
static __device__ int g_noalloc_err;

// Device addresses of the two arrays on the current device, looked up once
// per device (in host code their names are only host-side stand-ins).
struct NoallocAddr {
  float* scratch;
  int* err;
};
static bool noalloc_addr(int dev, NoallocAddr* out) {
  static NoallocAddr addr[128] = {};
  if (dev < 0 || dev >= 128) return false;
  if (!addr[dev].scratch) {
    void* p = nullptr;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&q, g_noalloc_err) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    addr[dev].err = static_cast<int*>(q);
    addr[dev].scratch = static_cast<float*>(p);
  }
  *out = addr[dev];
  return true;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" int gpt2_layernorm_backward_noalloc(float* dinp, float* dweight, float* dbias,
                                               float* dinp_colsum, const float* dout,
                                               const float* inp, const float* weight,
                                               const float* mean, const float* rstd, int32_t N,
                                               int32_t C, void* cuda_stream) {
  if (!dinp || !dweight || !dbias || !dout || !inp || !weight || !mean || !rstd) {
    set_global_error("gpt2_layernorm_backward_noalloc: NULL pointer");
    return GPT2_ERR_ARG;
  }
  if (N < 1 || C < 4 || C > 1024 || C % 4 != 0) {
    set_global_error("gpt2_layernorm_backward_noalloc: need N >= 1, 4 <= C <= 1024, C % 4 == 0");
    return GPT2_ERR_ARG;
  }
  // rows move by bulk copies and columns by 16-byte vectors
  if (!aligned16(dinp) || !aligned16(dweight) || !aligned16(dbias) || !aligned16(dinp_colsum) ||
      !aligned16(dout) || !aligned16(inp) || !aligned16(weight) ||
      (reinterpret_cast<uintptr_t>(mean) & 3u) || (reinterpret_cast<uintptr_t>(rstd) & 3u)) {
    set_global_error("gpt2_layernorm_backward_noalloc: dinp, dweight, dbias, dinp_colsum, dout, inp "
                     "and weight need 16-byte aligned addresses, mean and rstd 4-byte");
    return GPT2_ERR_ARG;
  }
  const int64_t need = ln_partial_floats(N, C);
  if (need > NOALLOC_SCRATCH_FLOATS) {
    set_global_error("gpt2_layernorm_backward_noalloc: ceil(N/64)*3*C exceeds the 2^21-float "
                     "static scratch (N*C must stay below about 44.7 million)");
    return GPT2_ERR_ARG;
  }
  int dev = 0;
  NoallocAddr a = {};
  if (cudaGetDevice(&dev) != cudaSuccess || !noalloc_addr(dev, &a)) {
    cudaGetLastError();
    set_global_error("gpt2_layernorm_backward_noalloc: no device address for the static arrays");
    return GPT2_ERR_CUDA;
  }
  int64_t launches = 0;
  LaunchCtx c;
  c.stream = static_cast<cudaStream_t>(cuda_stream);
  c.err = a.err;
  c.launches = &launches;
  c.num_sms = 0;
  c.host_fail = 0;
  // No programmatic overlap with whatever the caller enqueued before (the
  // kernel reads weight before its dependency wait, which is only safe
  // behind the model's own kernels).
  c.pdl = 0;
  launch_layernorm_bwd<float>(c, dinp, nullptr, dweight, dbias, dinp_colsum, dout, inp, weight,
                              mean, rstd, N, C, true, a.scratch);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || c.host_fail) {
    set_global_error(e != cudaSuccess ? cudaGetErrorString(e) : "gpt2_layernorm_backward_noalloc: launch failed");
    return GPT2_ERR_CUDA;
  }
  return GPT2_OK;
}

extern "C" int gpt2_noalloc_check(void* cuda_stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  int dev = 0;
  NoallocAddr a = {};
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e != cudaSuccess || !noalloc_addr(dev, &a)) {
    cudaGetLastError();
    set_global_error(e != cudaSuccess ? cudaGetErrorString(e) : "gpt2_noalloc_check: no error word");
    return GPT2_ERR_CUDA;
  }
  int v = 0;
  e = cudaMemcpy(&v, a.err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_global_error(cudaGetErrorString(e));
    return GPT2_ERR_CUDA;
  }
  if (v) {
    cudaMemset(a.err, 0, sizeof(int));
    set_global_error("gpt2_noalloc_check: a bounded device wait expired");
    return GPT2_ERR_TIMEOUT;
  }
  return GPT2_OK;
}

// ============================================================ error path
// One warp waits on a freshly initialised mbarrier that nothing arrives
// on; the bounded wait (common.cuh) gives up after its time limit, records
// DEVERR_TIMEOUT and the kernel returns.
__global__ void expire_wait_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, err);
}

void launch_expire_wait(LaunchCtx& c) {
  expire_wait_kernel<<<1, 32, 0, c.stream>>>(c.err);
  (*c.launches)++;
}
