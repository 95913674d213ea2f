// k_gemm_tc.cu -- bf16 matmul on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// out[m, n] = sum_k A(m,k) B(n,k), fp32 accumulation, the three layouts of a
// Linear layer (GeekNews, "Implementing the neural-network layers": a matrix
// product plus a bias tiled over the rows): forward x W^T, data gradient
// dy W, weight gradient dy^T x.  Each operand is K-major or M/N-major in
// global memory and is copied as-is by TMA into 128-byte-swizzled shared
// memory, where the tcgen05 matrix descriptor states its major-ness -- no
// transposed copies are ever made.
//
// Persistent kernel: one CTA per SM walks the output tiles (split, m-tile,
// n-tile) of 128 x BN (BN = 128 or 256) in a grouped raster (GROUP_M m-tiles
// per sweep over n, so concurrently resident tiles share operands in L2).
//   warp 0      TMA producer: a ring of STAGES stages of 64 K-elements,
//               full/empty mbarriers
//   warp 1      allocates 2 x BN TMEM columns (two accumulators), one thread
//               issues tcgen05.mma (M=128, N=BN, K=16) and commits each stage
//               back to the producer and each finished tile to the epilogue
//   warps 2..9  epilogue, overlapping the next tile's MMAs: warp w reads its
//               TMEM lane quarter (w % 4: 32 rows) and column half
//               ((w-2)/4), 32-row x 128-byte chunks at a time.  Every global
//               byte of the epilogue moves by TMA: the chunk's auxiliary
//               input (residual stream, GELU derivative) is TMA-loaded
//               into a 128B-swizzled staging buffer, each thread (one row)
//               applies the fused epilogue from registers, writes the result
//               back into the staging buffer and one lane TMA-stores it (or
//               TMA-reduce-adds it, for the weight gradient's dW += ...).
// Every mbarrier wait is bounded (common.cuh); nothing traps.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <cstdio>
#include <cstring>

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

// 2-D tensor [outer][inner] (fp32 or bf16, row stride ld elements) or, with
// d2 > 1, 3-D [d2][outer][inner] (plane stride outer*ld); box {box_inner,
// box_outer, 1}; 128-byte swizzle; out-of-range reads are 0 and
// out-of-range writes are dropped.
static bool make_tmap(CUtensorMap* m, const void* base, bool f32, uint64_t inner, uint64_t outer,
                      uint64_t ld, uint32_t box_inner, uint32_t box_outer, uint64_t d2 = 1) {
  const uint64_t esz = f32 ? 4 : 2;
  cuuint64_t dims[3] = {inner, outer, d2};
  cuuint64_t strides[2] = {ld * esz, outer * ld * esz};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  d2 > 1 ? 3 : 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define TC_BM 128
#define TC_BK 64
#define GROUP_M 8
#define SPLITK_SERIAL_MAX 4
#define EPI_WARPS 8
#define TC_THREADS (64 + 32 * EPI_WARPS)
#define STG_BYTES 4096  // one epilogue chunk: 32 rows x 128 bytes, swizzled

template <int BN>
struct TcCfg {
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;
  static constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr size_t STAGING = (size_t)EPI_WARPS * STG_BYTES;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + STAGING + 1024 + 256;
};

__host__ __device__ constexpr uint32_t tc_idesc(int N, bool a_mn, bool b_mn) {
  return tc_idesc_bf16(TC_BM, N, a_mn, b_mn);
}

struct TileCoord {
  int split, mt, nt;
};
__device__ __forceinline__ TileCoord tile_coord(int t, int mtiles, int ntiles, int gm) {
  TileCoord c;
  const int per = mtiles * ntiles;
  c.split = t / per;
  const int r = t - c.split * per;
  const int group = r / (gm * ntiles);
  const int first_m = group * gm;
  const int gsize = min(mtiles - first_m, gm);
  const int idx = r - group * gm * ntiles;
  c.mt = first_m + idx % gsize;
  c.nt = idx / gsize;
  return c;
}

// Byte offset of 16-byte chunk c of row r in a 128B-swizzled staging buffer.
__device__ __forceinline__ uint32_t stg_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void put8_bf16(uint8_t* p, const float* v) {
  uint4 u;
  __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]), t1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 t2 = __floats2bfloat162_rn(v[4], v[5]), t3 = __floats2bfloat162_rn(v[6], v[7]);
  u.x = *reinterpret_cast<uint32_t*>(&t0);
  u.y = *reinterpret_cast<uint32_t*>(&t1);
  u.z = *reinterpret_cast<uint32_t*>(&t2);
  u.w = *reinterpret_cast<uint32_t*>(&t3);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void get8_bf16(const uint8_t* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

struct EpiMaps {
  CUtensorMap out, out2, aux;
};

// The bias of the warp's BN/2 columns of a tile, 4 per lane (lane l holds
// columns 4l..4l+3 of the half), loaded before the accumulator is waited
// for so that the global-load latency is hidden; read back by shuffles.
template <int BN>
__device__ __forceinline__ float4 load_bias4(const GemmArgs& g, bool use_bias, int n0, int half, int lane) {
  float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
  const int n = n0 + half * (BN / 2) + 4 * lane;
  if (!use_bias || 4 * lane >= BN / 2) return b;
  if (n + 4 <= g.N) return *reinterpret_cast<const float4*>(g.bias + n);
  if (n < g.N) b.x = g.bias[n];
  if (n + 1 < g.N) b.y = g.bias[n + 1];
  if (n + 2 < g.N) b.z = g.bias[n + 2];
  return b;
}

// gelu(x) and gelu'(x) (tanh form) of 8 values, in f32x2 pairs with one
// tanh.approx per value.  With S = sqrt(2/pi), A = 0.044715, x2 = x^2,
// th = tanh(x (S + S A x2)), h = (1 + th)/2 and m = (1 - th)/2:
//   gelu(x)  = x h
//   gelu'(x) = h + x (1 - th^2) (S/2 + 3 S A x2/2) = h + (x (2S + 6 S A x2)) (h m)
// since 1 - th^2 = 4 h m.
__device__ __forceinline__ void gelu8_f2(const float* x, float* gl, float* gd) {
  const uint64_t c_sa = f2_pack(GELU_S * GELU_A, GELU_S * GELU_A), c_s = f2_pack(GELU_S, GELU_S);
  const uint64_t c_h = f2_pack(0.5f, 0.5f), c_nh = f2_pack(-0.5f, -0.5f);
  const uint64_t c_sa6 = f2_pack(6.f * GELU_S * GELU_A, 6.f * GELU_S * GELU_A), c_s2 = f2_pack(2.f * GELU_S, 2.f * GELU_S);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint64_t xx = f2_pack(x[i], x[i + 1]);
    const uint64_t x2 = f2_mul(xx, xx);
    float z0, z1;
    f2_unpack(f2_mul(xx, f2_fma(x2, c_sa, c_s)), z0, z1);
    const uint64_t th = f2_pack(tanh_hw(z0), tanh_hw(z1));
    const uint64_t h = f2_fma(th, c_h, c_h), m = f2_fma(th, c_nh, c_h);
    f2_unpack(f2_mul(xx, h), gl[i], gl[i + 1]);
    f2_unpack(f2_fma(f2_mul(xx, f2_fma(x2, c_sa6, c_s2)), f2_mul(h, m), h), gd[i], gd[i + 1]);
  }
}

// EPI_DOT_AUX: minus the dot product of row m's 64 columns from n (one
// attention head) into dot_out[(b * (N / 64) + n / 64) * dot_T + t],
// m = b * dot_T + t
__device__ __forceinline__ void store_dot(const GemmArgs& g, int m, int n, float dot) {
  if (m < g.M) {
    const int b = m / g.dot_T, t = m - b * g.dot_T;
    g.dot_out[((int64_t)b * (g.N >> 6) + (n >> 6)) * g.dot_T + t] = -dot;
  }
}

// Epilogue of one accumulator tile for one epilogue warp: 32 rows (this
// warp's TMEM lane quarter, global rows mrow..mrow+31) by the warp's column
// half of the BN columns starting at n0.  taddr: TMEM address of the
// accumulator at (lane quarter, column 0); bq: load_bias4 of the tile.
// The fp32 arithmetic runs in f32x2 pairs: the warps of lane quarter 1
// share a scheduler with the thread that issues the MMAs, and packed
// instructions take half the issue slots of scalar ones.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& g, const EpiMaps& em, uint8_t* stg,
                                              uint64_t* abar, uint32_t& aux_phase, uint32_t taddr0,
                                              int half, int lane, int mrow, int n0, int split_idx,
                                              bool split, bool f32, bool has_aux, bool use_bias,
                                              float4 bq, int* err, int* tflag = nullptr, int nsplits = 1,
                                              uint8_t* stg2 = nullptr) {
  const int epi = g.epi;
  const int CW = f32 ? 32 : 64;  // columns per 128-byte staging row
  if (tflag) {
    // split-K reduced in the kernel: split s of this warp's region adds its
    // part into the output only after split s-1 has (ld.acquire of the
    // region's flag), so the sum is formed in split order -- deterministic
    if (lane == 0) {
      flag_wait(tflag, split_idx, err);
      fence_proxy_async_global();
    }
    __syncwarp();
  }
#pragma unroll 1
  for (int cc = half * (BN / 2); cc < (half + 1) * (BN / 2); cc += CW) {
    const int ncol = n0 + cc;
    if (ncol >= g.N) break;
    if (lane == 0) bulk_wait_read0();  // staging no longer read by earlier stores
    __syncwarp();
    if (has_aux && lane == 0) {
      mbar_arrive_expect_tx(abar, STG_BYTES);
      tma_load_2d(stg, &em.aux, abar, ncol, mrow);
    }
    float v[64];
    const uint32_t taddr = taddr0 + (uint32_t)cc;
    {
      uint32_t r[32];
      tmem_ld32(taddr, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
      if (!f32) {
        tmem_ld32(taddr + 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j++) v[32 + j] = __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 32; j < 64; j++) v[j] = 0.f;
      }
    }
    if (g.dequant_a) {  // E4M3 products: undo the operands' per-tensor scales
      const float sc = 1.f / (*g.dequant_a * *g.dequant_b);
#pragma unroll
      for (int j = 0; j < 64; j++) v[j] *= sc;
    }
    if (use_bias) {
      const int lb = (cc - half * (BN / 2)) >> 2;  // lane holding this chunk's first 4 columns
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        if (j < CW) {
          const int src = lb + (j >> 2);
          const float b0 = __shfl_sync(0xffffffffu, bq.x, src), b1 = __shfl_sync(0xffffffffu, bq.y, src);
          const float b2 = __shfl_sync(0xffffffffu, bq.z, src), b3 = __shfl_sync(0xffffffffu, bq.w, src);
          f2_unpack(f2_add(f2_pack(v[j], v[j + 1]), f2_pack(b0, b1)), v[j], v[j + 1]);
          f2_unpack(f2_add(f2_pack(v[j + 2], v[j + 3]), f2_pack(b2, b3)), v[j + 2], v[j + 3]);
        }
      }
    }
    if (has_aux) {
      mbar_wait(abar, aux_phase, err);
      aux_phase ^= 1u;
    }
    float dot = 0.f;  // EPI_DOT_AUX
    // results (and the auxiliary input) in the thread's staging row
    if (f32) {
#pragma unroll
      for (int c = 0; c < 8; c++) {
        float4* p = reinterpret_cast<float4*>(stg + stg_off(lane, c));
        float4 o = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        if (has_aux) {  // EPI_RESIDUAL: out = residual + (acc + bias)
          const float4 r = *p;
          f2_unpack(f2_add(f2_pack(r.x, r.y), f2_pack(o.x, o.y)), o.x, o.y);
          f2_unpack(f2_add(f2_pack(r.z, r.w), f2_pack(o.z, o.w)), o.z, o.w);
        }
        *p = o;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 8; c++) {
        uint8_t* p = stg + stg_off(lane, c);
        float o[8];
        if (has_aux) {  // EPI_MUL_AUX: out = acc * aux; EPI_DOT_AUX: out = acc, dot += out * aux
          float hv[8];
          get8_bf16(p, hv);
          if (epi == EPI_DOT_AUX) {
#pragma unroll
            for (int q = 0; q < 8; q++) {
              o[q] = v[8 * c + q];
              dot = fmaf(__bfloat162float(__float2bfloat16_rn(o[q])), hv[q], dot);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; q += 2)
              f2_unpack(f2_mul(f2_pack(v[8 * c + q], v[8 * c + q + 1]), f2_pack(hv[q], hv[q + 1])), o[q], o[q + 1]);
          }
        } else if (epi == EPI_GELU_FWD && !split) {  // out = gelu'(x); v keeps gelu(x) for out2
          {
            float gl[8];
            gelu8_f2(&v[8 * c], gl, o);
#pragma unroll
            for (int q = 0; q < 8; q++) v[8 * c + q] = gl[q];
          }
          if (stg2) put8_bf16(stg2 + stg_off(lane, c), &v[8 * c]);  // gelu(x) into the second buffer
        } else {
#pragma unroll
          for (int q = 0; q < 8; q++) o[q] = v[8 * c + q];
        }
        put8_bf16(p, o);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (split) tma_store_3d(&em.out, stg, ncol, mrow, split_idx);
      else if (epi == EPI_ACCUM) tma_reduce_add_2d(&em.out, stg, ncol, mrow);
      else tma_store_2d(&em.out, stg, ncol, mrow);
      if (epi == EPI_GELU_FWD && !split && stg2) tma_store_2d(&em.out2, stg2, ncol, mrow);
      bulk_commit();
    }
    if (epi == EPI_DOT_AUX) store_dot(g, mrow + lane, ncol, dot);
    if (g.colsum_out && !f32 && !split) {
      // column sums of the stored values over the warp's 32 rows, read back
      // from the staging rows (lane l: columns 2l, 2l+1 of the chunk)
      uint64_t s01 = f2_pack(0.f, 0.f);
      const int ch = lane >> 2, wo = (lane & 3) * 4;
#pragma unroll 8
      for (int r = 0; r < 32; r++) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(stg + r * 128 + ((ch ^ (r & 7)) << 4) + wo);
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
        s01 = f2_add(s01, f2_pack(f.x, f.y));
      }
      float s0, s1;
      f2_unpack(s01, s0, s1);
      const int n = ncol + 2 * lane;
      if (mrow < g.M && n < g.N)
        *reinterpret_cast<float2*>(g.colsum_out + (int64_t)(mrow >> 5) * g.N + n) = make_float2(s0, s1);
    }
    if (epi == EPI_GELU_FWD && !split && !stg2) {  // second output: gelu(x), already in v
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 8; c++) {
        float o[8];
#pragma unroll
        for (int q = 0; q < 8; q++) o[q] = v[8 * c + q];
        put8_bf16(stg + stg_off(lane, c), o);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&em.out2, stg, ncol, mrow);
        bulk_commit();
      }
    }
  }
  if (tflag) {  // this split's additions are complete: hand the region on
    if (lane == 0) {
      bulk_wait0();
      fence_proxy_async_global();
      st_release_gpu(tflag, split_idx + 1 == nsplits ? 0 : split_idx + 1);
    }
    __syncwarp();
  }
}

struct EpiFlags {
  bool split, f32, has_aux, use_bias;
};
__device__ __forceinline__ EpiFlags epi_flags(const GemmArgs& g, int splits) {
  EpiFlags f;
  const int epi = g.epi;
  f.split = splits > 1;
  f.f32 = f.split || epi == EPI_RESIDUAL || epi == EPI_ACCUM || (epi == EPI_STORE && g.out_f32);
  f.has_aux = !f.split && (epi == EPI_RESIDUAL || epi == EPI_MUL_AUX || epi == EPI_DOT_AUX);
  f.use_bias = !f.split && g.bias && (epi == EPI_STORE || epi == EPI_GELU_FWD || epi == EPI_RESIDUAL);
  return f;
}

// Epilogue of a tile whose result combines the accumulator with an
// auxiliary input tile of the same shape (EPI_RESIDUAL: fp32 residual
// stream; EPI_MUL_AUX: bf16 gelu'), with the aux tiles fetched
// ahead: the warp owns two staging buffers used by alternate chunks; the
// caller issues chunk 0's aux load into buffer 0 before it waits for the
// accumulator, and chunk c+1's load goes into the other buffer while chunk
// c is processed.  The result overwrites the aux tile in place and is
// TMA-stored from there.  aph: phase bits of the two aux barriers.
template <int BN>
__device__ __forceinline__ void epilogue_tile_aux(const GemmArgs& g, const EpiMaps& em, uint8_t* stg2,
                                                  uint64_t* abar2, uint32_t& aph, uint32_t taddr0,
                                                  int half, int lane, int mrow, int n0, bool f32,
                                                  bool use_bias, float4 bq, int* err) {
  const int CW = f32 ? 32 : 64;  // columns per 128-byte staging row
  const int nch = (BN / 2) / CW;
#pragma unroll 1
  for (int c = 0; c < nch; c++) {
    const int cc = half * (BN / 2) + c * CW;
    const int ncol = n0 + cc;
    if (ncol >= g.N) break;
    uint8_t* stg = stg2 + (c & 1) * STG_BYTES;
    if (c + 1 < nch && ncol + CW < g.N) {
      if (lane == 0) bulk_wait_read0();  // the other buffer's last store has read it
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&abar2[(c + 1) & 1], STG_BYTES);
        tma_load_2d(stg2 + ((c + 1) & 1) * STG_BYTES, &em.aux, &abar2[(c + 1) & 1], ncol + CW, mrow);
      }
    }
    float v[64];
    const uint32_t taddr = taddr0 + (uint32_t)cc;
    {
      uint32_t r[32];
      tmem_ld32(taddr, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
      if (!f32) {
        tmem_ld32(taddr + 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j++) v[32 + j] = __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 32; j < 64; j++) v[j] = 0.f;
      }
    }
    if (use_bias) {
      const int lb = (cc - half * (BN / 2)) >> 2;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        if (j < CW) {
          const int src = lb + (j >> 2);
          const float b0 = __shfl_sync(0xffffffffu, bq.x, src), b1 = __shfl_sync(0xffffffffu, bq.y, src);
          const float b2 = __shfl_sync(0xffffffffu, bq.z, src), b3 = __shfl_sync(0xffffffffu, bq.w, src);
          f2_unpack(f2_add(f2_pack(v[j], v[j + 1]), f2_pack(b0, b1)), v[j], v[j + 1]);
          f2_unpack(f2_add(f2_pack(v[j + 2], v[j + 3]), f2_pack(b2, b3)), v[j + 2], v[j + 3]);
        }
      }
    }
    mbar_wait(&abar2[c & 1], (aph >> (c & 1)) & 1u, err);
    aph ^= 1u << (c & 1);
    float dot = 0.f;  // EPI_DOT_AUX
    if (f32) {  // EPI_RESIDUAL: out = residual + (acc + bias)
#pragma unroll
      for (int q = 0; q < 8; q++) {
        float4* pp = reinterpret_cast<float4*>(stg + stg_off(lane, q));
        const float4 r = *pp;
        float4 o;
        f2_unpack(f2_add(f2_pack(r.x, r.y), f2_pack(v[4 * q], v[4 * q + 1])), o.x, o.y);
        f2_unpack(f2_add(f2_pack(r.z, r.w), f2_pack(v[4 * q + 2], v[4 * q + 3])), o.z, o.w);
        *pp = o;
      }
    } else {  // EPI_MUL_AUX: out = acc * aux
#pragma unroll
      for (int q = 0; q < 8; q++) {
        uint8_t* pp = stg + stg_off(lane, q);
        float hv[8], o[8];
        get8_bf16(pp, hv);
        if (g.epi == EPI_DOT_AUX) {  // out = acc, dot += out * aux
#pragma unroll
          for (int k = 0; k < 8; k++) {
            o[k] = v[8 * q + k];
            dot = fmaf(__bfloat162float(__float2bfloat16_rn(o[k])), hv[k], dot);
          }
        } else {  // EPI_MUL_AUX: out = acc * aux
#pragma unroll
          for (int k = 0; k < 8; k += 2)
            f2_unpack(f2_mul(f2_pack(v[8 * q + k], v[8 * q + k + 1]), f2_pack(hv[k], hv[k + 1])), o[k], o[k + 1]);
        }
        put8_bf16(pp, o);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&em.out, stg, ncol, mrow);
      bulk_commit();
    }
    if (g.epi == EPI_DOT_AUX) store_dot(g, mrow + lane, ncol, dot);
    if (g.colsum_out && !f32) {
      uint64_t s01 = f2_pack(0.f, 0.f);
      const int ch = lane >> 2, wo = (lane & 3) * 4;
#pragma unroll 8
      for (int r = 0; r < 32; r++) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(stg + r * 128 + ((ch ^ (r & 7)) << 4) + wo);
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
        s01 = f2_add(s01, f2_pack(f.x, f.y));
      }
      float s0, s1;
      f2_unpack(s01, s0, s1);
      const int n = ncol + 2 * lane;
      if (mrow < g.M && n < g.N)
        *reinterpret_cast<float2*>(g.colsum_out + (int64_t)(mrow >> 5) * g.N + n) = make_float2(s0, s1);
    }
  }
}

template <int BN, bool A_K, bool B_K>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ EpiMaps em, GemmArgs g, int k_tiles, int k_per_split,
                   int splits, int* flags, int* err) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* staging = smem + (size_t)S * Cfg::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;      // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint64_t* aux_bar = acc_empty + 2;   // [EPI_WARPS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_bar + EPI_WARPS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtiles = (g.M + TC_BM - 1) / TC_BM, ntiles = (g.N + BN - 1) / BN;
  const int total = splits * mtiles * ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; a++) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], EPI_WARPS); }
    for (int w = 0; w < EPI_WARPS; w++) mbar_init(&aux_bar[w], 1);
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
  pdl_trigger();  // dependents launch only once every CTA holds its tensor memory
  pdl_wait();  // from here on global memory written by the previous kernel is read

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;  // running k-tile counter over all tiles of this CTA
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, mtiles, ntiles, GROUP_M);
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
        const TileCoord tc = tile_coord(t, mtiles, ntiles, GROUP_M);
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
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2, quarter = warp & 3, half = ew >> 2;
    // flags: split-K reduced in the kernel (the epilogue then accumulates like a
    // single split, in split order); else split s writes partial plane s
    const EpiFlags f = epi_flags(g, flags ? 1 : splits);
    uint32_t aux_phase = 0;
    int ti = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ti++) {
      const TileCoord tc = tile_coord(t, mtiles, ntiles, GROUP_M);
      const int a = ti & 1;
      int* tflag = flags ? flags + (int64_t)(tc.mt * ntiles + tc.nt) * EPI_WARPS + ew : nullptr;
      const float4 bq = load_bias4<BN>(g, f.use_bias, tc.nt * BN, half, lane);
      mbar_wait(&acc_full[a], (uint32_t)(ti >> 1) & 1u, err);
      tc_fence_after();
      epilogue_tile<BN>(g, em, staging + (size_t)ew * STG_BYTES, &aux_bar[ew], aux_phase,
                        tmem + (uint32_t)(a * BN) + ((uint32_t)(quarter * 32) << 16), half, lane,
                        tc.mt * TC_BM + quarter * 32, tc.nt * BN, tc.split, f.split, f.f32, f.has_aux,
                        f.use_bias, bq, err, tflag, splits);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
    }
    if (lane == 0) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

// ------------------------------------------------------------ CTA-pair kernel
// Output tiles of 256 x 256 per cluster of two CTAs on one TPC (M = 256
// tcgen05 MMA, cta_group::2).  CTA r of the pair loads rows 128r..128r+127
// of the tile's A rows and of its B rows (output columns), so a stage is
// 32 KB per CTA instead of 48 KB for a 128 x 256 tile on one SM: the ring
// is six stages deep, and each SM pulls a third fewer operand bytes through
// L2 per flop.  Both CTAs' TMA loads complete on the leader's (rank 0) full
// barrier; the leader's single MMA thread multicasts each stage's release
// and each finished accumulator to both CTAs; both CTAs' epilogue warps
// release an accumulator on the leader's barrier.  Each CTA drains its own
// 128 accumulator lanes with the epilogue above.
#define PAIR_BN 256
#define GROUP_PAIRS 4
// AUX: two staging buffers per warp, for one operand stage: an epilogue that
// reads an aux tile (EPI_RESIDUAL, EPI_MUL_AUX) fetches it ahead into one,
// and the GELU forward writes its two outputs into both at once.
template <bool AUX>
struct PairCfgT {
  static constexpr int STAGES = AUX ? 5 : 6;
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;            // 128 rows of A
  static constexpr uint32_t B_BYTES = (PAIR_BN / 2) * TC_BK * 2;     // 128 rows of B
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr size_t STAGING = (size_t)EPI_WARPS * STG_BYTES * (AUX ? 2 : 1);
  // + 1024 alignment slack + 512 for the barriers (up to 32) and the TMEM slot
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + STAGING + 1024 + 512;
};

// F8: A and B are E4M3 codes (one byte each, K-major), the MMA kind is
// f8f6f4 and a 128-byte smem row holds 128 K-elements, so a stage covers
// K = 128 with the same byte layout and descriptors as 64 bf16.
template <bool A_K, bool B_K, bool AUX, bool F8 = false>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ EpiMaps em, GemmArgs g, int k_tiles, int k_per_split,
                        int splits, int* flags, int* err) {
  using PairCfg = PairCfgT<AUX>;
  constexpr int S = PairCfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* staging = smem + (size_t)S * PairCfg::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + PairCfg::STAGING);  // used in the leader
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;      // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2], used in the leader
  uint64_t* aux_bar = acc_empty + 2;   // [EPI_WARPS][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_bar + 2 * EPI_WARPS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int mpairs = (g.M + 2 * TC_BM - 1) / (2 * TC_BM), ntiles = (g.N + PAIR_BN - 1) / PAIR_BN;
  const int total = splits * mpairs * ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; a++) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], 2 * EPI_WARPS); }
    for (int w = 0; w < 2 * EPI_WARPS; w++) mbar_init(&aux_bar[w], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 2 * PAIR_BN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();  // dependents launch only once every CTA holds its tensor memory
  pdl_wait();  // from here on global memory written by the previous kernel is read

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;  // running k-tile counter over all tiles of this pair
      for (int t = pair; t < total; t += npairs) {
        const TileCoord tc = tile_coord(t, mpairs, ntiles, GROUP_PAIRS);
        const int m0 = (2 * tc.mt + (int)rank) * TC_BM;
        const int nb0 = tc.nt * PAIR_BN + (int)rank * (PAIR_BN / 2);
        const int kt0 = tc.split * k_per_split;
        const int nkt = min(k_tiles, kt0 + k_per_split) - kt0;
        for (int i = 0; i < nkt; i++, it++) {
          const int s = it % S;
          const uint32_t ph = (uint32_t)(it / S) & 1u;
          mbar_wait(&empty[s], ph ^ 1u, err);
          uint8_t* sa = smem + (size_t)s * PairCfg::STAGE_BYTES;
          uint8_t* sb = sa + PairCfg::A_BYTES;
          const uint32_t bar = cluster_addr(&full[s], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * PairCfg::STAGE_BYTES);
          const int k = (kt0 + i) * (F8 ? 2 * TC_BK : TC_BK);
          if (A_K) {
            tma_load_2d_pair(sa, &tmA, bar, k, m0);
          } else {
            tma_load_2d_pair(sa, &tmA, bar, m0, k);
            tma_load_2d_pair(sa + 8192, &tmA, bar, m0 + 64, k);
          }
          if (B_K) {
            tma_load_2d_pair(sb, &tmB, bar, k, nb0);
          } else {
            tma_load_2d_pair(sb, &tmB, bar, nb0, k);
            tma_load_2d_pair(sb + 8192, &tmB, bar, nb0 + 64, k);
          }
        }
      }
      // every release the leader will still multicast here has landed
      for (int d = max(0, it - S); d < it; d++) mbar_wait(&empty[d % S], (uint32_t)(d / S) & 1u, err);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = F8 ? tc_idesc_e4m3(2 * TC_BM, PAIR_BN) : tc_idesc_bf16(2 * TC_BM, PAIR_BN, !A_K, !B_K);
      int it = 0, ti = 0;
      for (int t = pair; t < total; t += npairs, ti++) {
        const TileCoord tc = tile_coord(t, mpairs, ntiles, GROUP_PAIRS);
        const int kt0 = tc.split * k_per_split;
        const int nkt = min(k_tiles, kt0 + k_per_split) - kt0;
        const int a = ti & 1;
        mbar_wait(&acc_empty[a], ((uint32_t)(ti >> 1) & 1u) ^ 1u, err);
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(a * PAIR_BN);
        for (int i = 0; i < nkt; i++, it++) {
          const int s = it % S;
          const uint32_t ph = (uint32_t)(it / S) & 1u;
          mbar_wait(&full[s], ph, err);
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + (size_t)s * PairCfg::STAGE_BYTES);
          const uint32_t b0 = a0 + PairCfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; kk++) {
            const uint64_t ad = A_K ? sw128_desc(a0 + kk * 32, 16, 1024) : sw128_desc(a0 + kk * 2048, 8192, 1024);
            const uint64_t bd = B_K ? sw128_desc(b0 + kk * 32, 16, 1024) : sw128_desc(b0 + kk * 2048, 8192, 1024);
            if (F8) tc_mma_e4m3_pair(acc, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
            else tc_mma_bf16_pair(acc, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit_pair_both(&empty[s]);
        }
        tc_commit_pair_both(&acc_full[a]);
      }
      // both CTAs' epilogues have released every accumulator
      for (int d = max(0, ti - 2); d < ti; d++) mbar_wait(&acc_empty[d & 1], (uint32_t)(d >> 1) & 1u, err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2, quarter = warp & 3, half = ew >> 2;
    const EpiFlags f = epi_flags(g, flags ? 1 : splits);  // flags: split-K reduced in the kernel
    uint32_t aux_phase = 0;
    int ti = 0;
    for (int t = pair; t < total; t += npairs, ti++) {
      const TileCoord tc = tile_coord(t, mpairs, ntiles, GROUP_PAIRS);
      const int a = ti & 1;
      int* tflag = flags ? flags + ((int64_t)(tc.mt * ntiles + tc.nt) * 2 + rank) * EPI_WARPS + ew : nullptr;
      const int mrow = (2 * tc.mt + (int)rank) * TC_BM + quarter * 32, n0 = tc.nt * PAIR_BN;
      const uint32_t taddr = tmem + (uint32_t)(a * PAIR_BN) + ((uint32_t)(quarter * 32) << 16);
      if (AUX && f.has_aux) {
        // chunk 0's aux tile, fetched while this tile's MMAs still run
        uint8_t* stg2 = staging + (size_t)ew * 2 * STG_BYTES;
        const int ncol0 = n0 + half * (PAIR_BN / 2);
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        if (lane == 0 && ncol0 < g.N) {
          mbar_arrive_expect_tx(&aux_bar[2 * ew], STG_BYTES);
          tma_load_2d(stg2, &em.aux, &aux_bar[2 * ew], ncol0, mrow);
        }
        const float4 bq = load_bias4<PAIR_BN>(g, f.use_bias, n0, half, lane);
        mbar_wait(&acc_full[a], (uint32_t)(ti >> 1) & 1u, err);
        tc_fence_after();
        epilogue_tile_aux<PAIR_BN>(g, em, stg2, &aux_bar[2 * ew], aux_phase, taddr, half, lane, mrow, n0,
                                   f.f32, f.use_bias, bq, err);
      } else {
        const float4 bq = load_bias4<PAIR_BN>(g, f.use_bias, n0, half, lane);
        mbar_wait(&acc_full[a], (uint32_t)(ti >> 1) & 1u, err);
        tc_fence_after();
        // with the doubled staging of the AUX configuration, the GELU
        // forward writes its two outputs into two buffers (no wait between)
        uint8_t* st = AUX ? staging + (size_t)ew * 2 * STG_BYTES : staging + (size_t)ew * STG_BYTES;
        epilogue_tile<PAIR_BN>(g, em, st, &aux_bar[2 * ew], aux_phase, taddr, half, lane, mrow, n0, tc.split,
                               f.split, f.f32, f.has_aux, f.use_bias, bq, err, tflag, splits,
                               AUX ? st + STG_BYTES : nullptr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&acc_empty[a], 0));
    }
    if (lane == 0) bulk_wait0();
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * PAIR_BN);
  }
}

// out[m, n] += sum over splits of partial[s][m][n], splits in order.
__global__ void splitk_reduce_kernel(float* out, int64_t ldo, const float* partial, int splits,
                                     int M, int N) {
  pdl_trigger();
  pdl_wait();
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
  EpiMaps em;
  memset(&em, 0, sizeof(em));
  bool ok;
  if (A_K) ok = make_tmap(&ta, g.A, false, g.K, g.M, g.lda, 64, TC_BM);
  else ok = make_tmap(&ta, g.A, false, g.M, g.K, g.lda, 64, 64);
  if (B_K) ok = ok && make_tmap(&tb, g.B, false, g.K, g.N, g.ldb, 64, BN);
  else ok = ok && make_tmap(&tb, g.B, false, g.N, g.K, g.ldb, 64, 64);
  const int k_tiles = (g.K + TC_BK - 1) / TC_BK;
  const int kps = (k_tiles + splits - 1) / splits;
  const int zs = (k_tiles + kps - 1) / kps;
  const int64_t nflags = (int64_t)((g.M + TC_BM - 1) / TC_BM) * ((g.N + BN - 1) / BN) * EPI_WARPS;
  // in-kernel reduction for up to SPLITK_SERIAL_MAX splits (each split waits
  // for the previous one, ~3 us per hand-off); more splits use partial planes
  int* flags = zs > 1 && zs <= SPLITK_SERIAL_MAX && g.splitk_flags && nflags <= g.splitk_flag_count ? g.splitk_flags
                                                                                                       : nullptr;
  if (zs > 1 && !flags) {
    ok = ok && make_tmap(&em.out, partial, true, g.N, g.M, g.N, 32, 32, zs);
  } else {
    const bool f32 = g.epi == EPI_RESIDUAL || g.epi == EPI_ACCUM || (g.epi == EPI_STORE && g.out_f32);
    ok = ok && make_tmap(&em.out, g.out, f32, g.N, g.M, g.ldo, f32 ? 32 : 64, 32);
    if (g.epi == EPI_GELU_FWD) ok = ok && make_tmap(&em.out2, g.out2, false, g.N, g.M, g.ldo, 64, 32);
    if (g.epi == EPI_RESIDUAL) ok = ok && make_tmap(&em.aux, g.aux, true, g.N, g.M, g.ldo, 32, 32);
    if (g.epi == EPI_MUL_AUX || g.epi == EPI_DOT_AUX) ok = ok && make_tmap(&em.aux, g.aux, false, g.N, g.M, g.ldo, 64, 32);
  }
  if (!ok) {
    fprintf(stderr, "gpt2: tensor map encoding failed (M=%d N=%d K=%d)\n", g.M, g.N, g.K);
    c.host_fail = 1;
    return;
  }
  const int tiles = zs * ((g.N + BN - 1) / BN) * ((g.M + TC_BM - 1) / TC_BM);
  const int grid = std::min(tiles, c.num_sms);
  auto kern = gemm_tc_kernel<BN, A_K, B_K>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<BN>::SMEM);
  launch_pdl(c, kern, dim3(grid), dim3(TC_THREADS), TcCfg<BN>::SMEM, ta, tb, em, g, k_tiles, kps, zs, flags, c.err);
  if (zs > 1 && !flags) {
    const int64_t n4 = (int64_t)g.M * g.N / 4;
    int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)c.num_sms * 8);
    launch_pdl(c, splitk_reduce_kernel, dim3(blocks), dim3(256), 0, static_cast<float*>(g.out), g.ldo, partial, zs, g.M, g.N);
  }
}

template <bool A_K, bool B_K, bool AUX>
static void launch_tc_pair(LaunchCtx& c, const GemmArgs& g, int splits, float* partial) {
  CUtensorMap ta, tb;
  EpiMaps em;
  memset(&em, 0, sizeof(em));
  bool ok;
  if (A_K) ok = make_tmap(&ta, g.A, false, g.K, g.M, g.lda, 64, TC_BM);
  else ok = make_tmap(&ta, g.A, false, g.M, g.K, g.lda, 64, 64);
  if (B_K) ok = ok && make_tmap(&tb, g.B, false, g.K, g.N, g.ldb, 64, PAIR_BN / 2);
  else ok = ok && make_tmap(&tb, g.B, false, g.N, g.K, g.ldb, 64, 64);
  const int k_tiles = (g.K + TC_BK - 1) / TC_BK;
  const int kps = (k_tiles + splits - 1) / splits;
  const int zs = (k_tiles + kps - 1) / kps;
  const int64_t nflags = (int64_t)((g.M + 2 * TC_BM - 1) / (2 * TC_BM)) * ((g.N + PAIR_BN - 1) / PAIR_BN) * 2 * EPI_WARPS;
  // in-kernel reduction for up to SPLITK_SERIAL_MAX splits (each split waits
  // for the previous one, ~3 us per hand-off); more splits use partial planes
  int* flags = zs > 1 && zs <= SPLITK_SERIAL_MAX && g.splitk_flags && nflags <= g.splitk_flag_count ? g.splitk_flags
                                                                                                       : nullptr;
  if (zs > 1 && !flags) {
    ok = ok && make_tmap(&em.out, partial, true, g.N, g.M, g.N, 32, 32, zs);
  } else {
    const bool f32 = g.epi == EPI_RESIDUAL || g.epi == EPI_ACCUM || (g.epi == EPI_STORE && g.out_f32);
    ok = ok && make_tmap(&em.out, g.out, f32, g.N, g.M, g.ldo, f32 ? 32 : 64, 32);
    if (g.epi == EPI_GELU_FWD) ok = ok && make_tmap(&em.out2, g.out2, false, g.N, g.M, g.ldo, 64, 32);
    if (g.epi == EPI_RESIDUAL) ok = ok && make_tmap(&em.aux, g.aux, true, g.N, g.M, g.ldo, 32, 32);
    if (g.epi == EPI_MUL_AUX || g.epi == EPI_DOT_AUX) ok = ok && make_tmap(&em.aux, g.aux, false, g.N, g.M, g.ldo, 64, 32);
  }
  if (!ok) {
    fprintf(stderr, "gpt2: tensor map encoding failed (M=%d N=%d K=%d)\n", g.M, g.N, g.K);
    c.host_fail = 1;
    return;
  }
  using Cfg = PairCfgT<AUX>;
  auto kern = gemm_tc_pair_kernel<A_K, B_K, AUX>;
  static int max_pairs = 0;  // co-resident clusters of two, per instantiation
  if (max_pairs == 0) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * c.num_sms);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = c.num_sms / 2;
    }
    max_pairs = n;
  }
  const int pair_tiles = zs * ((g.N + PAIR_BN - 1) / PAIR_BN) * ((g.M + 2 * TC_BM - 1) / (2 * TC_BM));
  const int pairs = std::min(pair_tiles, max_pairs);
  launch_pdl_cluster(c, kern, dim3(2 * pairs), dim3(TC_THREADS), Cfg::SMEM, 2, ta, tb, em, g, k_tiles, kps, zs, flags, c.err);
  if (zs > 1 && !flags) {
    const int64_t n4 = (int64_t)g.M * g.N / 4;
    int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)c.num_sms * 8);
    launch_pdl(c, splitk_reduce_kernel, dim3(blocks), dim3(256), 0, static_cast<float*>(g.out), g.ldo, partial, zs, g.M, g.N);
  }
}

// ====================================================================== few-row products
// out[m, n] = sum_k A[m, k] W[n, k] (+ epilogue) for M <= 16 rows of A (one
// row per sequence while generating).  The operands swap roles: a CTA owns
// 128 weight rows n as the tcgen05 M dimension and the (up to 16) rows of A
// form the N = 16 dimension, so the MMA is M = 128, N = 16 and no tensor-core
// work is spent on padding rows; the weights stream once through TMA (the
// product is bound by HBM).  When there are few 128-row tiles, K is split
// over a cluster of up to 8 CTAs; their fp32 partials are added by the first
// CTA of the cluster through distributed shared memory, in rank order, so the
// sum does not depend on scheduling.  Thread n of the epilogue owns weight row
// n and writes out[m, n] for every m: consecutive lanes, consecutive columns.
#define RT_STAGES 6
#define RT_XROWS 16
#define RT_WBYTES (TC_BM * 128)     // 128 weight rows x 64 bf16
#define RT_XBYTES (RT_XROWS * 128)  // 16 rows of A x 64 bf16
#define RT_THREADS 128
#define RT_SMEM (1024 + RT_STAGES * (RT_WBYTES + RT_XBYTES) + TC_BM * RT_XROWS * 4 + 256)
#define RT_MAX_CLUSTER 8

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__global__ void __launch_bounds__(RT_THREADS, 1)
    gemm_rows_tc_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                        const GemmArgs g, int ktiles, int kps, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sW = sm;                                                   // [STAGES][128 x 64]
  uint8_t* sX = sW + RT_STAGES * RT_WBYTES;                           // [STAGES][16 x 64]
  float* red = reinterpret_cast<float*>(sX + RT_STAGES * RT_XBYTES);  // [16][128] partial sums
  uint64_t* full = reinterpret_cast<uint64_t*>(red + TC_BM * RT_XROWS);
  uint64_t* empty = full + RT_STAGES;
  uint64_t* done = empty + RT_STAGES;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  const uint32_t S = cluster_size(), rank = cluster_rank();
  const int n0 = (int)(blockIdx.x / S) * TC_BM;
  const int kt0 = (int)rank * kps;
  const int nk = max(0, min(ktiles, kt0 + kps) - kt0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_STAGES; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tw);
    tma_prefetch_desc(&tx);
  }
  if (warp == 1) { tmem_alloc(tslot, 32); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_trigger();  // dependents launch only once every CTA holds its tensor memory
  pdl_wait();
  if (warp == 0 && lane == 0) {  // TMA producer
    for (int i = 0; i < nk; i++) {
      const int s = i % RT_STAGES;
      if (i >= RT_STAGES) mbar_wait(&empty[s], (uint32_t)((i / RT_STAGES) - 1) & 1u, err);
      mbar_arrive_expect_tx(&full[s], RT_WBYTES + RT_XBYTES);
      tma_load_2d(sW + s * RT_WBYTES, &tw, &full[s], (kt0 + i) * TC_BK, n0);
      tma_load_2d(sX + s * RT_XBYTES, &tx, &full[s], (kt0 + i) * TC_BK, 0);
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    const uint32_t idesc = tc_idesc_bf16(TC_BM, RT_XROWS, false, false);
    for (int i = 0; i < nk; i++) {
      const int s = i % RT_STAGES;
      mbar_wait(&full[s], (uint32_t)(i / RT_STAGES) & 1u, err);
      tc_fence_after();
      const uint32_t a = smem_u32(sW + s * RT_WBYTES), b = smem_u32(sX + s * RT_XBYTES);
#pragma unroll
      for (int kk = 0; kk < TC_BK / 16; kk++)
        tc_mma_bf16(tm, sw128_desc(a + kk * 32, 16, 1024), sw128_desc(b + kk * 32, 16, 1024), idesc,
                    (i > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    tc_commit(done);  // with no MMA issued it arrives at once
  }
  __syncwarp();
  mbar_wait(done, 0, err);
  tc_fence_after();
  float acc[RT_XROWS];
  const int nl = warp * 32 + lane;  // this thread's weight row within the tile
  if (nk > 0) {
    uint32_t r[32];
    tmem_ld32(tm + ((uint32_t)(warp * 32) << 16), r);
    tmem_ld_wait();
#pragma unroll
    for (int m = 0; m < RT_XROWS; m++) acc[m] = __uint_as_float(r[m]);
  } else {
#pragma unroll
    for (int m = 0; m < RT_XROWS; m++) acc[m] = 0.f;
  }
  if (S > 1) {
#pragma unroll
    for (int m = 0; m < RT_XROWS; m++) red[m * TC_BM + nl] = acc[m];
    cluster_sync();  // every rank's partial sums are in its shared memory
    if (rank == 0) {
      for (uint32_t q = 1; q < S; q++) {
        const uint32_t base = cluster_addr(red, q);
#pragma unroll
        for (int m = 0; m < RT_XROWS; m++) acc[m] += ld_cluster_f32(base + (uint32_t)(m * TC_BM + nl) * 4u);
      }
    }
    cluster_sync();  // the first CTA has read them: the others may exit
  }
  const int n = n0 + nl;
  if (rank == 0 && n < g.N) {
    const float bias = g.bias ? g.bias[n] : 0.f;
    const int64_t orow = g.out_row ? (int64_t)(*g.out_row) * g.out_row_stride : 0;
#pragma unroll
    for (int m = 0; m < RT_XROWS; m++) {
      if (m >= g.M) break;
      const float x = acc[m] + bias;
      const int64_t o = (int64_t)m * g.ldo + n;
      if (g.epi == EPI_RESIDUAL) {
        static_cast<float*>(g.out)[orow + o] = static_cast<const float*>(g.aux)[o] + x;
      } else if (g.epi == EPI_GELU_FWD) {
        float gl, gd;
        gelu_and_grad_hw(x, gl, gd);
        static_cast<bf16*>(g.out)[orow + o] = __float2bfloat16_rn(gd);
        static_cast<bf16*>(g.out2)[orow + o] = __float2bfloat16_rn(gl);
      } else if (g.out_f32) {
        static_cast<float*>(g.out)[orow + o] = x;
      } else {
        static_cast<bf16*>(g.out)[orow + o] = __float2bfloat16_rn(x);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) { tc_fence_after(); tmem_dealloc(tm, 32); }
}

bool gemm_rows_applies(const GemmArgs& g) {
  return g.M >= 1 && g.M <= RT_XROWS && g.a_kmajor && g.b_kmajor && !g.colsum_out &&
         (g.epi == EPI_STORE || g.epi == EPI_RESIDUAL || g.epi == EPI_GELU_FWD);
}

void launch_gemm_rows(LaunchCtx& c, const GemmArgs& g) {
  CUtensorMap tw, tx;
  bool ok = make_tmap(&tw, g.B, false, g.K, g.N, g.ldb, 64, TC_BM);
  ok = ok && make_tmap(&tx, g.A, false, g.K, g.M, g.lda, 64, RT_XROWS);
  if (!ok) {
    fprintf(stderr, "gpt2: tensor map encoding failed (M=%d N=%d K=%d)\n", g.M, g.N, g.K);
    c.host_fail = 1;
    return;
  }
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(gemm_rows_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RT_SMEM);
    attr = true;
  }
  const int ntiles = (g.N + TC_BM - 1) / TC_BM;
  const int ktiles = (g.K + TC_BK - 1) / TC_BK;
  // split K so that the clusters cover the SMs; no rank without K tiles
  int S = std::min({RT_MAX_CLUSTER, ktiles, std::max(1, (c.num_sms + ntiles - 1) / ntiles)});
  const int kps = (ktiles + S - 1) / S;
  S = (ktiles + kps - 1) / kps;
  if (S > 1)
    launch_pdl_cluster(c, gemm_rows_tc_kernel, dim3(ntiles * S), dim3(RT_THREADS), RT_SMEM, S, tw, tx, g, ktiles,
                       kps, c.err);
  else
    launch_pdl(c, gemm_rows_tc_kernel, dim3(ntiles), dim3(RT_THREADS), RT_SMEM, tw, tx, g, ktiles, kps, c.err);
}

// [outer][inner] bytes (E4M3 codes), row stride ld bytes, box {128, box_outer}.
static bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                         uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void launch_gemm_fp8(LaunchCtx& c, const GemmArgs& g) {
  CUtensorMap ta, tb;
  EpiMaps em;
  memset(&em, 0, sizeof(em));
  bool ok = g.epi == EPI_STORE && g.a_kmajor && g.b_kmajor && g.dequant_a && g.dequant_b;
  ok = ok && make_tmap_u8(&ta, g.A, g.K, g.M, g.lda, TC_BM);
  ok = ok && make_tmap_u8(&tb, g.B, g.K, g.N, g.ldb, PAIR_BN / 2);
  ok = ok && make_tmap(&em.out, g.out, g.out_f32, g.N, g.M, g.ldo, g.out_f32 ? 32 : 64, 32);
  if (!ok) {
    fprintf(stderr, "gpt2: fp8 matmul setup failed (M=%d N=%d K=%d)\n", g.M, g.N, g.K);
    c.host_fail = 1;
    return;
  }
  using Cfg = PairCfgT<false>;
  auto kern = gemm_tc_pair_kernel<true, true, false, true>;
  static int max_pairs = 0;
  if (max_pairs == 0) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * c.num_sms);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = c.num_sms / 2;
    }
    max_pairs = n;
  }
  const int k_tiles = (g.K + 2 * TC_BK - 1) / (2 * TC_BK);  // 128 codes per stage
  const int pair_tiles = ((g.N + PAIR_BN - 1) / PAIR_BN) * ((g.M + 2 * TC_BM - 1) / (2 * TC_BM));
  const int pairs = std::min(pair_tiles, max_pairs);
  launch_pdl_cluster(c, kern, dim3(2 * pairs), dim3(TC_THREADS), Cfg::SMEM, 2, ta, tb, em, g, k_tiles, k_tiles, 1,
                     (int*)nullptr, c.err);
}

void launch_gemm_bf16(LaunchCtx& c, const GemmArgs& g) {
  if (g.epi == EPI_DOT_AUX && (g.out_f32 || g.N % 64 != 0 || !g.aux || !g.dot_out || g.dot_T <= 0 ||
                               g.M % g.dot_T != 0)) {
    fprintf(stderr, "gpt2: EPI_DOT_AUX needs a bf16 output, N %% 64 == 0 and M a multiple of dot_T\n");
    c.host_fail = 1;
    return;
  }
  if (gemm_rows_applies(g)) {  // a few rows of A: the weights stream once, M and N swapped
    launch_gemm_rows(c, g);
    return;
  }
  if (g.out_row) {  // a device-side output row is a feature of the few-row kernel only
    c.host_fail = 1;
    return;
  }
  const int BN = g.N >= 256 ? 256 : 128;
  const int tiles = ((g.N + BN - 1) / BN) * ((g.M + TC_BM - 1) / TC_BM);
  const int k_tiles = (g.K + TC_BK - 1) / TC_BK;
  int splits = 1;
  if (g.epi == EPI_ACCUM && g.splitk_scratch && tiles < c.num_sms) {
    if (BN == 256) {
      // CTA pairs: as many splits as keep every pair busy in one wave (the
      // fewest hand-offs for the same balance)
      const int pair_tiles = ((g.N + PAIR_BN - 1) / PAIR_BN) * ((g.M + 2 * TC_BM - 1) / (2 * TC_BM));
      splits = std::max(1, std::min((c.num_sms / 2) / pair_tiles, k_tiles / 8));
    } else {
      splits = std::max(1, std::min((2 * c.num_sms) / tiles, k_tiles / 8));
    }
    while (splits > 1 && (int64_t)splits * g.M * g.N > g.splitk_scratch_floats) splits--;
  }
  float* partial = splits > 1 ? g.splitk_scratch : nullptr;
#define TC_DISPATCH(BNV)                                                     \
  if (g.a_kmajor && g.b_kmajor) launch_tc<BNV, true, true>(c, g, splits, partial);        \
  else if (g.a_kmajor && !g.b_kmajor) launch_tc<BNV, true, false>(c, g, splits, partial); \
  else if (!g.a_kmajor && g.b_kmajor) launch_tc<BNV, false, true>(c, g, splits, partial); \
  else launch_tc<BNV, false, false>(c, g, splits, partial);
  if (BN == 256) {
    // epilogues that read an aux tile use the prefetching variant; the model's
    // aux GEMMs (attproj / fcproj forward, fcproj dgrad) are A K-major
    const bool aux = splits == 1 && (g.epi == EPI_RESIDUAL || g.epi == EPI_MUL_AUX || g.epi == EPI_GELU_FWD ||
                                     g.epi == EPI_DOT_AUX);
    if (aux && g.a_kmajor && g.b_kmajor) launch_tc_pair<true, true, true>(c, g, splits, partial);
    else if (aux && g.a_kmajor) launch_tc_pair<true, false, true>(c, g, splits, partial);
    else if (g.a_kmajor && g.b_kmajor) launch_tc_pair<true, true, false>(c, g, splits, partial);
    else if (g.a_kmajor && !g.b_kmajor) launch_tc_pair<true, false, false>(c, g, splits, partial);
    else if (!g.a_kmajor && g.b_kmajor) launch_tc_pair<false, true, false>(c, g, splits, partial);
    else launch_tc_pair<false, false, false>(c, g, splits, partial);
  } else {
    TC_DISPATCH(128)
  }
#undef TC_DISPATCH
}
