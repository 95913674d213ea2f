// k_gemm_tc.cu -- bf16 matmul on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// out[m, n] = sum_k A(m,k) B(n,k), fp32 accumulation, the three layouts of a
// Linear layer's forward (x W^T), data gradient (dy W) and weight gradient
// (dy^T x) served by one kernel: each operand is either K-major or
// M/N-major in global memory and is copied as-is by TMA into 128-byte-
// swizzled shared memory, where the tcgen05 matrix descriptor states its
// major-ness -- no transposed copies are ever made.
//
// One CTA computes one 128 x BN output tile (BN = 128 or 256) over a range
// of K (the whole K, or one split of it for the weight gradient):
//   warp 0      TMA producer: a ring of STAGES shared-memory stages,
//               64 K-elements per stage, full/empty mbarriers;
//   warp 1      allocates BN TMEM columns, then one elected thread issues
//               tcgen05.mma (M=128, N=BN, K=16, four per stage) and commits
//               each stage back to the producer;
//   warps 2..5  epilogue: tcgen05.ld 32 rows x 32 columns at a time from the
//               warp's TMEM lane quarter, apply the fused epilogue (bias,
//               GELU, residual, GELU backward, accumulate) and store.
// Every mbarrier wait is bounded (see common.cuh); nothing traps.
#include <cuda.h>

#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "kernels.h"

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn g_encode = nullptr;

bool gemm_bf16_init() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return true;
}

// 2-D bf16 tensor [outer][inner] with row stride ld elements; box
// {box_inner, box_outer}; 128-byte swizzle; out-of-range elements read 0.
static bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define TC_BM 128
#define TC_BK 64

template <int BN>
struct TcCfg {
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;
  static constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;  // + align + barriers
};

__host__ __device__ constexpr uint32_t tc_idesc(int N, bool a_mn, bool b_mn) {
  return tc_idesc_bf16(TC_BM, N, a_mn, b_mn);
}

__device__ __forceinline__ void store8_bf16(bf16* p, const float* v) {
  uint4 u;
  __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]), t1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 t2 = __floats2bfloat162_rn(v[4], v[5]), t3 = __floats2bfloat162_rn(v[6], v[7]);
  u.x = *reinterpret_cast<uint32_t*>(&t0);
  u.y = *reinterpret_cast<uint32_t*>(&t1);
  u.z = *reinterpret_cast<uint32_t*>(&t2);
  u.w = *reinterpret_cast<uint32_t*>(&t3);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void load8_bf16(const bf16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// Epilogue for 8 consecutive columns n..n+7 of row m (all in range when
// full8, else element-wise bounds).
__device__ __forceinline__ void epi8(const GemmArgs& g, float* v, int m, int n, bool full8,
                                     float* partial) {
  const int64_t o = (int64_t)m * g.ldo + n;
  if (partial) {  // split-K: raw partial sums, fp32, leading dimension N
    float* p = partial + (int64_t)m * g.N + n;
    if (full8) {
      *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      for (int j = 0; j < 8; j++) if (n + j < g.N) p[j] = v[j];
    }
    return;
  }
  if (g.bias && g.epi != EPI_GELU_BWD && g.epi != EPI_ACCUM) {
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] += (full8 || n + j < g.N) ? g.bias[n + j] : 0.f;
  }
  switch (g.epi) {
    case EPI_STORE:
      if (g.out_f32) {
        float* p = static_cast<float*>(g.out) + o;
        if (full8) {
          *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
        } else {
          for (int j = 0; j < 8; j++) if (n + j < g.N) p[j] = v[j];
        }
      } else {
        bf16* p = static_cast<bf16*>(g.out) + o;
        if (full8) store8_bf16(p, v);
        else for (int j = 0; j < 8; j++) if (n + j < g.N) p[j] = __float2bfloat16_rn(v[j]);
      }
      break;
    case EPI_BIAS_GELU: {
      bf16* p = static_cast<bf16*>(g.out) + o;
      bf16* q = static_cast<bf16*>(g.out2) + o;
      float gv[8];
#pragma unroll
      for (int j = 0; j < 8; j++) gv[j] = gelu_f(v[j]);
      if (full8) { store8_bf16(p, v); store8_bf16(q, gv); }
      else for (int j = 0; j < 8; j++) if (n + j < g.N) { p[j] = __float2bfloat16_rn(v[j]); q[j] = __float2bfloat16_rn(gv[j]); }
    } break;
    case EPI_RESIDUAL: {
      float* p = static_cast<float*>(g.out) + o;
      const float* r = static_cast<const float*>(g.aux) + o;
      if (full8) {
        const float4 a = *reinterpret_cast<const float4*>(r);
        const float4 b = *reinterpret_cast<const float4*>(r + 4);
        *reinterpret_cast<float4*>(p) = make_float4(a.x + v[0], a.y + v[1], a.z + v[2], a.w + v[3]);
        *reinterpret_cast<float4*>(p + 4) = make_float4(b.x + v[4], b.y + v[5], b.z + v[6], b.w + v[7]);
      } else {
        for (int j = 0; j < 8; j++) if (n + j < g.N) p[j] = r[j] + v[j];
      }
    } break;
    case EPI_GELU_BWD: {
      bf16* p = static_cast<bf16*>(g.out) + o;
      const bf16* h = static_cast<const bf16*>(g.aux) + o;
      if (full8) {
        float hv[8];
        load8_bf16(h, hv);
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] *= gelu_grad_f(hv[j]);
        store8_bf16(p, v);
      } else {
        for (int j = 0; j < 8; j++)
          if (n + j < g.N) p[j] = __float2bfloat16_rn(v[j] * gelu_grad_f(__bfloat162float(h[j])));
      }
    } break;
    case EPI_ACCUM: {
      float* p = static_cast<float*>(g.out) + o;
      if (full8) {
        float4 a = *reinterpret_cast<float4*>(p);
        float4 b = *reinterpret_cast<float4*>(p + 4);
        a.x += v[0]; a.y += v[1]; a.z += v[2]; a.w += v[3];
        b.x += v[4]; b.y += v[5]; b.z += v[6]; b.w += v[7];
        *reinterpret_cast<float4*>(p) = a;
        *reinterpret_cast<float4*>(p + 4) = b;
      } else {
        for (int j = 0; j < 8; j++) if (n + j < g.N) p[j] += v[j];
      }
    } break;
  }
}

// Persistent kernel: one CTA per SM walks the output tiles (split, m-tile,
// n-tile) in a grouped raster (GROUP_M m-tiles per column sweep, so the
// concurrently resident tiles share A and B tiles in L2).  Two TMEM
// accumulators let the epilogue of one tile run while the MMAs of the next
// one are issued.
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocation + MMA issuer (one thread)
//   warps 2..9  epilogue: warp w reads TMEM lane quarter w % 4, column half
//               (w - 2) / 4 of the tile
#define GROUP_M 8
#define EPI_WARPS 8
#define TC_THREADS (64 + 32 * EPI_WARPS)

struct TileCoord {
  int split, mt, nt;
};
__device__ __forceinline__ TileCoord tile_coord(int t, int mtiles, int ntiles) {
  TileCoord c;
  const int per = mtiles * ntiles;
  c.split = t / per;
  const int r = t - c.split * per;
  const int group = r / (GROUP_M * ntiles);
  const int first_m = group * GROUP_M;
  const int gsize = min(mtiles - first_m, GROUP_M);
  const int idx = r - group * GROUP_M * ntiles;
  c.mt = first_m + idx % gsize;
  c.nt = idx / gsize;
  return c;
}

template <int BN, bool A_K, bool B_K>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   GemmArgs g, int k_tiles, int k_per_split, int splits, float* partial, int* err) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * Cfg::STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;   // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtiles = (g.M + TC_BM - 1) / TC_BM, ntiles = (g.N + BN - 1) / BN;
  const int total = splits * mtiles * ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; a++) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], EPI_WARPS); }
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;  // running k-tile counter over all tiles of this CTA
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, mtiles, ntiles);
        const int m0 = tc.mt * TC_BM, n0 = tc.nt * BN;
        const int kt0 = tc.split * k_per_split;
        const int nkt = min(k_tiles, kt0 + k_per_split) - kt0;
        for (int i = 0; i < nkt; i++, it++) {
          const int s = it % S;
          const uint32_t ph = (uint32_t)(it / S) & 1u;
          mbar_wait(&empty[s], ph ^ 1u, err);
          uint8_t* sa = smem + (size_t)s * Cfg::STAGE_BYTES;
          uint8_t* sb = sa + Cfg::A_BYTES;
          mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
          const int k = (kt0 + i) * TC_BK;
          if (A_K) {
            tma_load_2d(sa, &tmA, &full[s], k, m0);
          } else {
            tma_load_2d(sa, &tmA, &full[s], m0, k);
            tma_load_2d(sa + 8192, &tmA, &full[s], m0 + 64, k);
          }
          if (B_K) {
            tma_load_2d(sb, &tmB, &full[s], k, n0);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; j++) tma_load_2d(sb + j * 8192, &tmB, &full[s], n0 + 64 * j, k);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc(BN, !A_K, !B_K);
      int it = 0, ti = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ti++) {
        const TileCoord tc = tile_coord(t, mtiles, ntiles);
        const int kt0 = tc.split * k_per_split;
        const int nkt = min(k_tiles, kt0 + k_per_split) - kt0;
        const int a = ti & 1;
        mbar_wait(&acc_empty[a], ((uint32_t)(ti >> 1) & 1u) ^ 1u, err);
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(a * BN);
        for (int i = 0; i < nkt; i++, it++) {
          const int s = it % S;
          const uint32_t ph = (uint32_t)(it / S) & 1u;
          mbar_wait(&full[s], ph, err);
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + (size_t)s * Cfg::STAGE_BYTES);
          const uint32_t b0 = a0 + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; kk++) {
            const uint64_t ad = A_K ? sw128_desc(a0 + kk * 32, 16, 1024) : sw128_desc(a0 + kk * 2048, 8192, 1024);
            const uint64_t bd = B_K ? sw128_desc(b0 + kk * 32, 16, 1024) : sw128_desc(b0 + kk * 2048, 8192, 1024);
            tc_mma_bf16(acc, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[a]);
      }
    }
  } else {
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    int ti = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ti++) {
      const TileCoord tc = tile_coord(t, mtiles, ntiles);
      const int m0 = tc.mt * TC_BM, n0 = tc.nt * BN;
      const int a = ti & 1;
      mbar_wait(&acc_full[a], (uint32_t)(ti >> 1) & 1u, err);
      tc_fence_after();
      const int m = m0 + quarter * 32 + lane;
      float* part = partial ? partial + (size_t)tc.split * (size_t)g.M * (size_t)g.N : nullptr;
#pragma unroll 1
      for (int cc = half * (BN / 2); cc < (half + 1) * (BN / 2); cc += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + (uint32_t)(a * BN) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)cc, r);
        tmem_ld_wait();
        if (m < g.M && n0 + cc < g.N) {
#pragma unroll
          for (int j0 = 0; j0 < 32; j0 += 8) {
            const int n = n0 + cc + j0;
            if (n >= g.N) break;
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; j++) v[j] = __uint_as_float(r[j0 + j]);
            epi8(g, v, m, n, n + 8 <= g.N, part);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

// out[m, n] += sum over splits of partial[s][m][n], splits in order.
__global__ void splitk_reduce_kernel(float* out, int64_t ldo, const float* partial, int splits,
                                     int M, int N) {
  const int64_t total = (int64_t)M * N;
  const int64_t MN = total;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total / 4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i * 4;
    const int64_t m = e / N, n = e % N;
    float4 s = *reinterpret_cast<const float4*>(partial + e);
    for (int k = 1; k < splits; k++) {
      const float4 v = *reinterpret_cast<const float4*>(partial + (int64_t)k * MN + e);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    float4* d = reinterpret_cast<float4*>(out + m * ldo + n);
    float4 o = *d;
    o.x += s.x; o.y += s.y; o.z += s.z; o.w += s.w;
    *d = o;
  }
}

template <int BN, bool A_K, bool B_K>
static void launch_tc(LaunchCtx& c, const GemmArgs& g, int splits, float* partial) {
  CUtensorMap ta, tb;
  bool ok;
  if (A_K) ok = make_tmap(&ta, g.A, g.K, g.M, g.lda, 64, TC_BM);
  else ok = make_tmap(&ta, g.A, g.M, g.K, g.lda, 64, 64);
  if (B_K) ok = ok && make_tmap(&tb, g.B, g.K, g.N, g.ldb, 64, BN);
  else ok = ok && make_tmap(&tb, g.B, g.N, g.K, g.ldb, 64, 64);
  if (!ok) {
    fprintf(stderr, "gpt2: tensor map encoding failed (M=%d N=%d K=%d)\n", g.M, g.N, g.K);
    c.host_fail = 1;
    return;
  }
  const int k_tiles = (g.K + TC_BK - 1) / TC_BK;
  const int kps = (k_tiles + splits - 1) / splits;
  const int zs = (k_tiles + kps - 1) / kps;
  const int tiles = zs * ((g.N + BN - 1) / BN) * ((g.M + TC_BM - 1) / TC_BM);
  const int grid = std::min(tiles, c.num_sms);
  auto kern = gemm_tc_kernel<BN, A_K, B_K>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<BN>::SMEM);
  kern<<<grid, TC_THREADS, TcCfg<BN>::SMEM, c.stream>>>(ta, tb, g, k_tiles, kps, zs, zs > 1 ? partial : nullptr, c.err);
  (*c.launches)++;
  if (zs > 1) {
    const int64_t n4 = (int64_t)g.M * g.N / 4;
    int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)c.num_sms * 8);
    splitk_reduce_kernel<<<blocks, 256, 0, c.stream>>>(static_cast<float*>(g.out), g.ldo, partial, zs, g.M, g.N);
    (*c.launches)++;
  }
}

void launch_gemm_bf16(LaunchCtx& c, const GemmArgs& g) {
  const int BN = g.N >= 256 ? 256 : 128;
  const int tiles = ((g.N + BN - 1) / BN) * ((g.M + TC_BM - 1) / TC_BM);
  const int k_tiles = (g.K + TC_BK - 1) / TC_BK;
  int splits = 1;
  if (g.epi == EPI_ACCUM && g.splitk_scratch && tiles < c.num_sms) {
    splits = std::max(1, std::min((2 * c.num_sms) / tiles, k_tiles / 8));
    while (splits > 1 && (int64_t)splits * g.M * g.N > g.splitk_scratch_floats) splits--;
  }
  float* partial = splits > 1 ? g.splitk_scratch : nullptr;
#define TC_DISPATCH(BNV)                                                     \
  if (g.a_kmajor && g.b_kmajor) launch_tc<BNV, true, true>(c, g, splits, partial);        \
  else if (g.a_kmajor && !g.b_kmajor) launch_tc<BNV, true, false>(c, g, splits, partial); \
  else if (!g.a_kmajor && g.b_kmajor) launch_tc<BNV, false, true>(c, g, splits, partial); \
  else launch_tc<BNV, false, false>(c, g, splits, partial);
  if (BN == 256) { TC_DISPATCH(256) } else { TC_DISPATCH(128) }
#undef TC_DISPATCH
}
