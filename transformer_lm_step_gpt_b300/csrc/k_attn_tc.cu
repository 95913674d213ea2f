// k_attn_tc.cu -- causal multi-head self-attention on the tcgen05 tensor cores.
//
// GeekNews, "A GPT-2-based ChatGPT clone in 3000 bytes of C", section "The
// Transformer core": per head, S = q k^T (scaled by 1/sqrt(hs)), the lower-
// triangular causal mask, softmax over each query row, times v.  Here the
// T x T score matrix is never stored: it is computed one 128 x 128 tile at a
// time in TMEM and folded into an online softmax (forward) or recomputed from
// the saved row logsumexp (backward).
//
// Head size 64.  Every tile of q, k, v, dy is one TMA box [128 rows x 64]
// of a 3-D tensor map over [B, T, width] (rows past T read as zero), landing
// 128-byte-swizzled in shared memory, where a tcgen05 descriptor can read it
// either as a K-major operand (rows = M or N) or as an MN-major one (rows =
// K) -- so S = q k^T, P v, dV = P^T dy, dK = dS^T q and dQ = dS k all read the
// same tiles.  P and dS are written to shared memory in the same swizzled
// K-major layout by the softmax threads.
//
//   forward   one CTA per (128-query block, batch*head), 8 warps: S -> TMEM,
//             row max / exp / row sum from TMEM (thread = query row), P -> smem,
//             O_blk = P v -> TMEM, O accumulated in registers with the
//             online-softmax rescale.  Saves lse = max + log(sum).
//   backward  D = rowsum(dy * y); one CTA per (128-key block, b*h) for dK, dV
//             (S^T, dP^T recomputed, dV += P^T dy, dK += dS^T q accumulated in
//             TMEM); one CTA per (128-query block, b*h) for dQ (dQ += dS k).
//             No atomics: every output element is written by one CTA, so the
//             result is deterministic.
// All mbarrier waits are bounded (common.cuh); a wait that gives up records
// a timeout and the kernel runs to completion without trapping.
#include <cuda.h>

#include <cstdio>

#include "common.cuh"
#include "kernels.h"

typedef CUresult (*EncodeTiledFnA)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnA encoder_fn() {
  static EncodeTiledFnA fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnA>(p);
  }
  return fn;
}

// [B][T][W] bf16 tensor, box {64, rows, 1}, 128-byte swizzle, rows past T zero.
static bool make_tmap_btw(CUtensorMap* m, const void* base, int B, int T, int W, int rows = 128) {
  EncodeTiledFnA f = encoder_fn();
  if (!f) return false;
  cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)W * 2, (cuuint64_t)T * W * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define AT_BLK 128
#define AT_HS 64
#define AT_TILE 16384u  // bytes of one [128 x 64] bf16 tile
#define AB_SUB 64
#define AT_SUBTILE 8192u  // bytes of one [64 x 64] bf16 tile

// descriptors of a [128 rows x 64] tile read as a K-major operand (rows = M
// or N, K = 64 head dims) at K-step kk (16 dims), or as an MN-major operand
// (rows = K, 64 columns = N) at K-step kk (16 rows)
__device__ __forceinline__ uint64_t kmaj(uint32_t tile, int kk) { return sw128_desc(tile + kk * 32, 16, 1024); }
__device__ __forceinline__ uint64_t mnmaj(uint32_t tile, int kk) { return sw128_desc(tile + kk * 2048, 8192, 1024); }
// descriptor of a [128 rows x 128] K-major operand stored as two 64-wide atoms
__device__ __forceinline__ uint64_t kmaj2(uint32_t buf, int kk) {
  return sw128_desc(buf + (kk >> 2) * AT_TILE + (kk & 3) * 32, 16, 1024);
}

// Write 8 consecutive bf16 values (columns c8*8 .. c8*8+7) of row r into a
// [128 x 128] K-major swizzled buffer (two 64-column atoms).
__device__ __forceinline__ void st_swz8(uint8_t* buf, int r, int c8, const float* v) {
  const int atom = c8 >> 3, chunk = (c8 & 7) ^ (r & 7);
  uint4 u;
  __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]), t1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 t2 = __floats2bfloat162_rn(v[4], v[5]), t3 = __floats2bfloat162_rn(v[6], v[7]);
  u.x = *reinterpret_cast<uint32_t*>(&t0);
  u.y = *reinterpret_cast<uint32_t*>(&t1);
  u.z = *reinterpret_cast<uint32_t*>(&t2);
  u.w = *reinterpret_cast<uint32_t*>(&t3);
  *reinterpret_cast<uint4*>(buf + atom * AT_TILE + r * 128 + chunk * 16) = u;
}

// Same as st_swz8 for a [128 x 64] buffer (one atom), given the row's base
// pointer (buf + r*128) and its swizzle (r & 7).
__device__ __forceinline__ void st_row8(uint8_t* rowp, int rx, int c8, const float* v) {
  uint4 u;
  __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]), t1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 t2 = __floats2bfloat162_rn(v[4], v[5]), t3 = __floats2bfloat162_rn(v[6], v[7]);
  u.x = *reinterpret_cast<uint32_t*>(&t0);
  u.y = *reinterpret_cast<uint32_t*>(&t1);
  u.z = *reinterpret_cast<uint32_t*>(&t2);
  u.w = *reinterpret_cast<uint32_t*>(&t3);
  *reinterpret_cast<uint4*>(rowp + ((c8 ^ rx) << 4)) = u;
}

// Backward elementwise step for 32 score columns of one row, from the TMEM
// words of S (rs) and dP (rd):  p = 2^(s*sl2 - lse2),  ds = p (dp - D).
// KEYROW: the row is a key and the columns are queries (dK/dV kernel; lse2
// and D per column), else the row is a query (dQ kernel; per row).  MASK
// applies the causal mask (only on sub-blocks that cross the diagonal).
template <bool KEYROW, bool MASK>
__device__ __forceinline__ void bwd_elementwise(const uint32_t* rs, const uint32_t* rd, const float* lse2c,
                                                const float* dc, float lse2r, float dr, float sl2,
                                                int col0, int rowpos, uint8_t* prow, uint8_t* srow,
                                                int rx, int c8base) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    float lv[8], dv[8];
    if (KEYROW) {
      const float4 a = *reinterpret_cast<const float4*>(lse2c + g * 8);
      const float4 b = *reinterpret_cast<const float4*>(lse2c + g * 8 + 4);
      const float4 c = *reinterpret_cast<const float4*>(dc + g * 8);
      const float4 d = *reinterpret_cast<const float4*>(dc + g * 8 + 4);
      lv[0] = a.x; lv[1] = a.y; lv[2] = a.z; lv[3] = a.w; lv[4] = b.x; lv[5] = b.y; lv[6] = b.z; lv[7] = b.w;
      dv[0] = c.x; dv[1] = c.y; dv[2] = c.z; dv[3] = c.w; dv[4] = d.x; dv[5] = d.y; dv[6] = d.z; dv[7] = d.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; j++) { lv[j] = lse2r; dv[j] = dr; }
    }
    float p[8], ds[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      float pv = ex2_hw(__uint_as_float(rs[g * 8 + j]) * sl2 - lv[j]);
      if (MASK) {
        const int col = col0 + g * 8 + j;
        const bool ok = KEYROW ? col >= rowpos : col <= rowpos;
        pv = ok ? pv : 0.f;
      }
      p[j] = pv;
      ds[j] = pv * (__uint_as_float(rd[g * 8 + j]) - dv[j]);
    }
    if (KEYROW) st_row8(prow, rx, c8base + g, p);
    st_row8(srow, rx, c8base + g, ds);
  }
}

__device__ __forceinline__ void store_row64_bf16(bf16* dst, const float* v, float mul) {
#pragma unroll
  for (int i = 0; i < 64; i += 8) {
    uint4 u;
    __nv_bfloat162 t0 = __floats2bfloat162_rn(v[i] * mul, v[i + 1] * mul);
    __nv_bfloat162 t1 = __floats2bfloat162_rn(v[i + 2] * mul, v[i + 3] * mul);
    __nv_bfloat162 t2 = __floats2bfloat162_rn(v[i + 4] * mul, v[i + 5] * mul);
    __nv_bfloat162 t3 = __floats2bfloat162_rn(v[i + 6] * mul, v[i + 7] * mul);
    u.x = *reinterpret_cast<uint32_t*>(&t0);
    u.y = *reinterpret_cast<uint32_t*>(&t1);
    u.z = *reinterpret_cast<uint32_t*>(&t2);
    u.w = *reinterpret_cast<uint32_t*>(&t3);
    *reinterpret_cast<uint4*>(dst + i) = u;
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ void store_row32_bf16(bf16* dst, const float* v, float mul) {
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    uint4 u;
    __nv_bfloat162 t0 = __floats2bfloat162_rn(v[i] * mul, v[i + 1] * mul);
    __nv_bfloat162 t1 = __floats2bfloat162_rn(v[i + 2] * mul, v[i + 3] * mul);
    __nv_bfloat162 t2 = __floats2bfloat162_rn(v[i + 4] * mul, v[i + 5] * mul);
    __nv_bfloat162 t3 = __floats2bfloat162_rn(v[i + 6] * mul, v[i + 7] * mul);
    u.x = *reinterpret_cast<uint32_t*>(&t0);
    u.y = *reinterpret_cast<uint32_t*>(&t1);
    u.z = *reinterpret_cast<uint32_t*>(&t2);
    u.w = *reinterpret_cast<uint32_t*>(&t3);
    *reinterpret_cast<uint4*>(dst + i) = u;
  }
}

// 8 warps: warps w and w+4 read the same TMEM lane quarter (w % 4, i.e. the
// same 32 query or key rows) and split the 128 score columns (half = w / 4
// takes columns 64*half .. 64*half+63) and the 64 output head dims
// (32*half .. 32*half+31).
#define AT_THREADS 256

// ============================================================ forward
// One CTA per (128-query block, b*h), keys walked in 64-row sub-blocks with
// a two-deep software pipeline: the MMA S(j+1) = q k(j+1)^T runs while the
// warps do the softmax of S(j), and O_blk(j) = P(j) v(j) runs while they
// start on j+1 (its result is folded into the register accumulator one
// iteration later).  TMEM: S[0], S[1], O[0], O[1] (64 columns each), so two
// CTAs share an SM.
// Warps w and w+4 exchange their half-row maxima through a double-buffered
// array and a 64-thread named barrier; the softmax warps hand P to the
// MMA-issuing thread through an mbarrier, so no step waits for the whole CTA.
// smem: Q | K0 K1 | V0 V1 (64-row tiles) | P0 P1 ([128 x 64]) | row-max exchange [2][2][128] | barriers
#define AF_SMEM (1024 + AT_TILE + 4 * AT_SUBTILE + 2 * AT_TILE + 2048 + 256)

__global__ void __launch_bounds__(AT_THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                       const __grid_constant__ CUtensorMap tm_qkv64, bf16* y, float* lse, int T,
                       int C, int NH, float scale, int* err) {
  pdl_trigger();
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sQ = sm;
  uint8_t* sK = sm + AT_TILE;            // 2 stages of [64 x 64]
  uint8_t* sV = sK + 2 * AT_SUBTILE;     // 2 stages
  uint8_t* sP = sV + 2 * AT_SUBTILE;     // 2 x [128 x 64]
  float* red = reinterpret_cast<float*>(sP + 2 * AT_TILE);  // [2 iterations][2 halves][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * AT_TILE + 2048);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;  // [2]
  uint64_t* v_full = bars + 3;  // [2]
  uint64_t* s_done = bars + 5;  // [2]
  uint64_t* o_done = bars + 7;  // [2]
  uint64_t* p_ready = bars + 9;  // 8 warp arrivals per sub-block
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 10);

  const int nqb = gridDim.x;
  const int qb = nqb - 1 - blockIdx.x;  // longest rows first
  const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
  const int q0 = qb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane, q = q0 + row;
  const int nsub = (min(q0 + AT_BLK, T) + AB_SUB - 1) / AB_SUB;  // key sub-blocks up to the last query

  if (tid == 0) {
    for (int i = 0; i < 9; i++) mbar_init(&bars[i], 1);
    mbar_init(p_ready, AT_THREADS / 32);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_qkv64);
  }
  if (warp == 0) { tmem_alloc(tslot, 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_wait();  // from here on global memory written by the previous kernel is read
  const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;
  const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
  const uint32_t idO = tc_idesc_bf16(128, 64, false, true);

  if (tid == 0) {
    mbar_arrive_expect_tx(q_full, AT_TILE);
    tma_load_3d(sQ, &tm_qkv, q_full, h * AT_HS, q0, b);
    for (int s = 0; s < 2 && s < nsub; s++) {
      mbar_arrive_expect_tx(&k_full[s], AT_SUBTILE);
      tma_load_3d(sK + s * AT_SUBTILE, &tm_qkv64, &k_full[s], C + h * AT_HS, s * AB_SUB, b);
      mbar_arrive_expect_tx(&v_full[s], AT_SUBTILE);
      tma_load_3d(sV + s * AT_SUBTILE, &tm_qkv64, &v_full[s], 2 * C + h * AT_HS, s * AB_SUB, b);
    }
    // S(0)
    mbar_wait(q_full, 0, err);
    mbar_wait(&k_full[0], 0, err);
    tc_fence_after();
    const uint32_t aQ = smem_u32(sQ), bK = smem_u32(sK);
#pragma unroll
    for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tm, kmaj(aQ, kk), kmaj(bK, kk), idS, kk > 0);
    tc_commit(&s_done[0]);
  }
  const float sl2 = scale * 1.4426950408889634f;  // scores -> log2 units
  float m = -INFINITY, lpart = 0.f, alpha_prev = 1.f;
  float o[32];
#pragma unroll
  for (int i = 0; i < 32; i++) o[i] = 0.f;

  for (int j = 0; j < nsub; j++) {
    const int sb = j & 1;
    const uint32_t tS = tm + (uint32_t)(sb * 64), tO = tm + 128 + (uint32_t)(sb * 64);
    mbar_wait(&s_done[sb], (uint32_t)(j >> 1) & 1u, err);
    tc_fence_after();
    if (tid == 0) {
      // S(j) is done with K stage sb: refill it with K(j+2)
      if (j + 2 < nsub) {
        mbar_arrive_expect_tx(&k_full[sb], AT_SUBTILE);
        tma_load_3d(sK + sb * AT_SUBTILE, &tm_qkv64, &k_full[sb], C + h * AT_HS, (j + 2) * AB_SUB, b);
      }
      // issue S(j+1) into the other S buffer (its last reader was softmax(j-1))
      if (j + 1 < nsub) {
        const int nb = sb ^ 1;
        mbar_wait(&k_full[nb], (uint32_t)((j + 1) >> 1) & 1u, err);
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ), bK = smem_u32(sK + nb * AT_SUBTILE);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tm + (uint32_t)(nb * 64), kmaj(aQ, kk), kmaj(bK, kk), idS, kk > 0);
        tc_commit(&s_done[nb]);
      }
    }
    const int k0 = j * AB_SUB;
    const bool diag = k0 + AB_SUB - 1 > q0;
    uint32_t r[32];
    tmem_ld32(tS + lanebase + half * 32, r);
    tmem_ld_wait();
    // pass 1: max over this half's 32 columns, exchanged with the partner warp
    float mx = -INFINITY;
    if (diag) {
#pragma unroll
      for (int jj = 0; jj < 32; jj++)
        if (k0 + half * 32 + jj <= q) mx = fmaxf(mx, __uint_as_float(r[jj]));
    } else {
#pragma unroll
      for (int jj = 0; jj < 32; jj++) mx = fmaxf(mx, __uint_as_float(r[jj]));
    }
    float* rd = red + sb * 256;
    rd[half * 128 + row] = mx;
    named_bar_sync(1 + quarter, 64);  // warps quarter and quarter + 4
    const float mnew = fmaxf(m, fmaxf(rd[row], rd[128 + row]));
    const float alpha = ex2_hw((m - mnew) * sl2);
    const float mo = mnew * sl2;
    // pass 2: P = exp(scale (s - mnew)) -> smem P[sb] (bf16), partial row sum
    float sum = 0.f;
    uint8_t* P = sP + sb * AT_TILE;
    uint8_t* prow = P + row * 128;
    if (diag) {
#pragma unroll
      for (int g = 0; g < 4; g++) {
        float p[8];
#pragma unroll
        for (int jj = 0; jj < 8; jj++) {
          const float e = ex2_hw(__uint_as_float(r[g * 8 + jj]) * sl2 - mo);
          p[jj] = k0 + half * 32 + g * 8 + jj <= q ? e : 0.f;
          sum += p[jj];
        }
        st_row8(prow, row & 7, half * 4 + g, p);
      }
    } else {
#pragma unroll
      for (int g = 0; g < 4; g++) {
        float p[8];
#pragma unroll
        for (int jj = 0; jj < 8; jj++) {
          p[jj] = ex2_hw(__uint_as_float(r[g * 8 + jj]) * sl2 - mo);
          sum += p[jj];
        }
        st_row8(prow, row & 7, half * 4 + g, p);
      }
    }
    lpart = lpart * alpha + sum;
    m = mnew;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_ready);
    if (tid == 0) {
      mbar_wait(p_ready, (uint32_t)j & 1u, err);
      tc_fence_after();
      mbar_wait(&v_full[sb], (uint32_t)(j >> 1) & 1u, err);
      const uint32_t aP = smem_u32(P), bV = smem_u32(sV + sb * AT_SUBTILE);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tO, kmaj(aP, kk), mnmaj(bV, kk), idO, kk > 0);
      tc_commit(&o_done[sb]);
    }
    // fold in O_blk(j-1) (its MMA ran during this iteration's softmax)
    if (j > 0) {
      const int pb = sb ^ 1;
      mbar_wait(&o_done[pb], (uint32_t)((j - 1) >> 1) & 1u, err);
      tc_fence_after();
      uint32_t ro[32];
      tmem_ld32(tm + 128 + (uint32_t)(pb * 64) + lanebase + half * 32, ro);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; i++) o[i] = o[i] * alpha_prev + __uint_as_float(ro[i]);
      if (tid == 0 && j + 1 < nsub) {  // PV(j-1) is done with V stage pb: load V(j+1)
        mbar_arrive_expect_tx(&v_full[pb], AT_SUBTILE);
        tma_load_3d(sV + pb * AT_SUBTILE, &tm_qkv64, &v_full[pb], 2 * C + h * AT_HS, (j + 1) * AB_SUB, b);
      }
    }
    alpha_prev = alpha;
    tc_fence_before();
  }
  {  // the last O_blk
    const int pb = (nsub - 1) & 1;
    mbar_wait(&o_done[pb], (uint32_t)((nsub - 1) >> 1) & 1u, err);
    tc_fence_after();
    uint32_t ro[32];
    tmem_ld32(tm + 128 + (uint32_t)(pb * 64) + lanebase + half * 32, ro);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; i++) o[i] = o[i] * alpha_prev + __uint_as_float(ro[i]);
  }
  __syncthreads();
  red[half * 128 + row] = lpart;
  __syncthreads();
  const float l = red[row] + red[128 + row];
  if (q < T) {
    store_row32_bf16(y + ((int64_t)b * T + q) * C + h * AT_HS + half * 32, o, 1.f / l);
    if (half == 0) lse[(int64_t)bh * T + q] = m * scale + logf(l);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tm, 256); }
}

// ============================================================ backward: D
// D[b,h,t] = sum_i dy[b,t,h*64+i] * y[b,t,h*64+i]
__global__ void attn_bwd_dsum_kernel(float* dsum, const bf16* dy, const bf16* y, int B, int T,
                                     int C, int NH) {
  pdl_trigger();
  pdl_wait();
  const int64_t n = (int64_t)B * T * NH;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int h = (int)(i % NH);
    const int64_t bt = i / NH;
    const int t = (int)(bt % T), b = (int)(bt / T);
    const uint4* a = reinterpret_cast<const uint4*>(dy + bt * C + h * AT_HS);
    const uint4* c = reinterpret_cast<const uint4*>(y + bt * C + h * AT_HS);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const uint4 ua = a[k], uc = c[k];
      const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wc[4] = {uc.x, uc.y, uc.z, uc.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[j]));
        const float2 fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wc[j]));
        s += fa.x * fc.x + fa.y * fc.y;
      }
    }
    dsum[((int64_t)b * NH + h) * T + t] = s;
  }
}

// ============================================================ backward: dK, dV
// One CTA per (128-key block, b*h); the queries are walked in 64-row
// sub-blocks so that a CTA needs 256 TMEM columns and ~97 KB of shared
// memory and two CTAs share an SM (one's MMAs overlap the other's
// elementwise work).
// smem: K | V | Q0 Q1 | dO0 dO1 (64-row tiles) | P^T | dS^T ([128 x 64]) |
//       lse[64] D[64] | barriers
#define AKV_SMEM (1024 + 2 * AT_TILE + 4 * AT_SUBTILE + 2 * AT_TILE + 512 + 256)

__global__ void __launch_bounds__(AT_THREADS, 2)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_qkv64,
                           const __grid_constant__ CUtensorMap tm_dy64, bf16* dqkv, const float* lse,
                           const float* dsum, int T, int C, int NH, float scale, int* err) {
  pdl_trigger();
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sK = sm;
  uint8_t* sV = sm + AT_TILE;
  uint8_t* sQ = sm + 2 * AT_TILE;                   // 2 stages of [64 x 64]
  uint8_t* sD = sQ + 2 * AT_SUBTILE;                // dO, 2 stages
  uint8_t* sP = sD + 2 * AT_SUBTILE;                // P^T  [128 keys x 64 queries]
  uint8_t* sS = sP + AT_TILE;                       // dS^T [128 keys x 64 queries]
  float* sl = reinterpret_cast<float*>(sS + AT_TILE);  // lse[64] (log2 units)
  float* sdd = sl + 64;                                 // D[64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + AT_TILE + 512);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;  // [2]
  uint64_t* s_done = bars + 3;
  uint64_t* o_done = bars + 4;
  uint64_t* p_ready = bars + 5;  // 8 warp arrivals per sub-block
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 6);

  const int kb = (int)gridDim.x - 1 - (int)blockIdx.x;  // key block; longest first
  const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
  const int k0 = kb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane, key = k0 + row;
  const int nsub = (T - k0 + AB_SUB - 1) / AB_SUB;  // 64-query sub-blocks from k0 to T

  if (tid == 0) {
    for (int i = 0; i < 5; i++) mbar_init(&bars[i], 1);
    mbar_init(p_ready, AT_THREADS / 32);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_qkv64);
    tma_prefetch_desc(&tm_dy64);
  }
  if (warp == 0) { tmem_alloc(tslot, 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_wait();  // from here on global memory written by the previous kernel is read
  const uint32_t tS = tm, tdP = tm + 64, tdV = tm + 128, tdK = tm + 192;
  const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;

  if (tid == 0) {
    mbar_arrive_expect_tx(kv_full, 2 * AT_TILE);
    tma_load_3d(sK, &tm_qkv, kv_full, C + h * AT_HS, k0, b);
    tma_load_3d(sV, &tm_qkv, kv_full, 2 * C + h * AT_HS, k0, b);
    for (int s = 0; s < 2 && s < nsub; s++) {
      mbar_arrive_expect_tx(&q_full[s], 2 * AT_SUBTILE);
      tma_load_3d(sQ + s * AT_SUBTILE, &tm_qkv64, &q_full[s], h * AT_HS, k0 + s * AB_SUB, b);
      tma_load_3d(sD + s * AT_SUBTILE, &tm_dy64, &q_full[s], h * AT_HS, k0 + s * AB_SUB, b);
    }
  }
  const float sl2 = scale * 1.4426950408889634f;
  const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
  const uint32_t idO = tc_idesc_bf16(128, 64, false, true);

  for (int it = 0; it < nsub; it++) {
    const int q0 = k0 + it * AB_SUB;
    const int st = it & 1;
    const uint32_t ph = (uint32_t)(it >> 1) & 1u;
    if (tid < AB_SUB) {  // this sub-block's lse (log2 units) and D
      const int qq = q0 + tid;
      sl[tid] = qq < T ? lse[(int64_t)bh * T + qq] * 1.4426950408889634f : INFINITY;
      sdd[tid] = qq < T ? dsum[(int64_t)bh * T + qq] : 0.f;
    }
    if (tid == 0) {
      if (it == 0) mbar_wait(kv_full, 0, err);
      mbar_wait(&q_full[st], ph, err);
      tc_fence_after();
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      const uint32_t bQ = smem_u32(sQ + st * AT_SUBTILE), bD = smem_u32(sD + st * AT_SUBTILE);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tS, kmaj(aK, kk), kmaj(bQ, kk), idS, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdP, kmaj(aV, kk), kmaj(bD, kk), idS, kk > 0);
      tc_commit(s_done);
    }
    __syncthreads();  // lse / D of this sub-block visible
    mbar_wait(s_done, (uint32_t)it & 1u, err);
    tc_fence_after();
    const bool diag = q0 < k0 + AT_BLK;
    {
      uint32_t rs[32], rd[32];
      tmem_ld32(tS + lanebase + half * 32, rs);
      tmem_ld32(tdP + lanebase + half * 32, rd);
      tmem_ld_wait();
      if (diag)
        bwd_elementwise<true, true>(rs, rd, sl + half * 32, sdd + half * 32, 0.f, 0.f, sl2, q0 + half * 32,
                                    key, sP + row * 128, sS + row * 128, row & 7, half * 4);
      else
        bwd_elementwise<true, false>(rs, rd, sl + half * 32, sdd + half * 32, 0.f, 0.f, sl2, q0 + half * 32,
                                     key, sP + row * 128, sS + row * 128, row & 7, half * 4);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_ready);
    if (tid == 0) {
      mbar_wait(p_ready, (uint32_t)it & 1u, err);
      tc_fence_after();
      const uint32_t aP = smem_u32(sP), aS = smem_u32(sS);
      const uint32_t bQ = smem_u32(sQ + st * AT_SUBTILE), bD = smem_u32(sD + st * AT_SUBTILE);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdV, kmaj(aP, kk), mnmaj(bD, kk), idO, (it > 0 || kk > 0));
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdK, kmaj(aS, kk), mnmaj(bQ, kk), idO, (it > 0 || kk > 0));
      tc_commit(o_done);
    }
    mbar_wait(o_done, (uint32_t)it & 1u, err);
    tc_fence_after();
    if (tid == 0 && it + 2 < nsub) {
      mbar_arrive_expect_tx(&q_full[st], 2 * AT_SUBTILE);
      tma_load_3d(sQ + st * AT_SUBTILE, &tm_qkv64, &q_full[st], h * AT_HS, q0 + 2 * AB_SUB, b);
      tma_load_3d(sD + st * AT_SUBTILE, &tm_dy64, &q_full[st], h * AT_HS, q0 + 2 * AB_SUB, b);
    }
    // every thread has waited o_done: the P^T / dS^T / lse buffers are free
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const int64_t C3 = 3 * (int64_t)C;
  float v[32];
  {
    uint32_t r[32];
    tmem_ld32(tdV + lanebase + half * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
  }
  if (key < T) store_row32_bf16(dqkv + ((int64_t)b * T + key) * C3 + 2 * C + h * AT_HS + half * 32, v, 1.f);
  {
    uint32_t r[32];
    tmem_ld32(tdK + lanebase + half * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
  }
  if (key < T) store_row32_bf16(dqkv + ((int64_t)b * T + key) * C3 + C + h * AT_HS + half * 32, v, scale);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tm, 256); }
}

// ============================================================ backward: dQ
// One CTA per (128-query block, b*h), keys walked in 64-row sub-blocks
// (256 TMEM columns, ~81 KB shared memory: two CTAs per SM).
// smem: Q | dO | K0 K1 | V0 V1 (64-row tiles) | dS ([128 x 64]) | barriers
#define AQ_SMEM (1024 + 2 * AT_TILE + 4 * AT_SUBTILE + AT_TILE + 256)

__global__ void __launch_bounds__(AT_THREADS, 2)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                          const __grid_constant__ CUtensorMap tm_dy,
                          const __grid_constant__ CUtensorMap tm_qkv64, bf16* dqkv, const float* lse,
                          const float* dsum, int T, int C, int NH, float scale, int* err) {
  pdl_trigger();
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sQ = sm;
  uint8_t* sD = sm + AT_TILE;
  uint8_t* sK = sm + 2 * AT_TILE;    // 2 stages of [64 x 64]
  uint8_t* sV = sK + 2 * AT_SUBTILE; // 2 stages
  uint8_t* sS = sV + 2 * AT_SUBTILE; // dS [128 queries x 64 keys]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + AT_TILE);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;  // [2]
  uint64_t* s_done = bars + 3;
  uint64_t* o_done = bars + 4;
  uint64_t* p_ready = bars + 5;  // 8 warp arrivals per sub-block
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 6);

  const int nqb = gridDim.x;
  const int qb = nqb - 1 - blockIdx.x;
  const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
  const int q0 = qb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane, q = q0 + row;
  const int nsub = (min(q0 + AT_BLK, T) + AB_SUB - 1) / AB_SUB;  // key sub-blocks up to the last query

  if (tid == 0) {
    for (int i = 0; i < 5; i++) mbar_init(&bars[i], 1);
    mbar_init(p_ready, AT_THREADS / 32);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_dy);
    tma_prefetch_desc(&tm_qkv64);
  }
  if (warp == 0) { tmem_alloc(tslot, 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_wait();  // from here on global memory written by the previous kernel is read
  const uint32_t tS = tm, tdP = tm + 64, tdQ = tm + 128;
  const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;

  if (tid == 0) {
    mbar_arrive_expect_tx(q_full, 2 * AT_TILE);
    tma_load_3d(sQ, &tm_qkv, q_full, h * AT_HS, q0, b);
    tma_load_3d(sD, &tm_dy, q_full, h * AT_HS, q0, b);
    for (int s = 0; s < 2 && s < nsub; s++) {
      mbar_arrive_expect_tx(&kv_full[s], 2 * AT_SUBTILE);
      tma_load_3d(sK + s * AT_SUBTILE, &tm_qkv64, &kv_full[s], C + h * AT_HS, s * AB_SUB, b);
      tma_load_3d(sV + s * AT_SUBTILE, &tm_qkv64, &kv_full[s], 2 * C + h * AT_HS, s * AB_SUB, b);
    }
  }
  const float sl2 = scale * 1.4426950408889634f;
  const float my_lse = q < T ? lse[(int64_t)bh * T + q] * 1.4426950408889634f : INFINITY;
  const float my_d = q < T ? dsum[(int64_t)bh * T + q] : 0.f;
  const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
  const uint32_t idO = tc_idesc_bf16(128, 64, false, true);

  for (int kb = 0; kb < nsub; kb++) {
    const int st = kb & 1;
    const uint32_t ph = (uint32_t)(kb >> 1) & 1u;
    const int k0 = kb * AB_SUB;
    if (tid == 0) {
      if (kb == 0) mbar_wait(q_full, 0, err);
      mbar_wait(&kv_full[st], ph, err);
      tc_fence_after();
      const uint32_t aQ = smem_u32(sQ), aD = smem_u32(sD);
      const uint32_t bK = smem_u32(sK + st * AT_SUBTILE), bV = smem_u32(sV + st * AT_SUBTILE);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tS, kmaj(aQ, kk), kmaj(bK, kk), idS, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdP, kmaj(aD, kk), kmaj(bV, kk), idS, kk > 0);
      tc_commit(s_done);
    }
    mbar_wait(s_done, (uint32_t)kb & 1u, err);
    tc_fence_after();
    const bool diag = k0 + AB_SUB > q0;
    {
      uint32_t rs[32], rd[32];
      tmem_ld32(tS + lanebase + half * 32, rs);
      tmem_ld32(tdP + lanebase + half * 32, rd);
      tmem_ld_wait();
      if (diag)
        bwd_elementwise<false, true>(rs, rd, nullptr, nullptr, my_lse, my_d, sl2, k0 + half * 32, q,
                                     nullptr, sS + row * 128, row & 7, half * 4);
      else
        bwd_elementwise<false, false>(rs, rd, nullptr, nullptr, my_lse, my_d, sl2, k0 + half * 32, q,
                                      nullptr, sS + row * 128, row & 7, half * 4);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_ready);
    if (tid == 0) {
      mbar_wait(p_ready, (uint32_t)kb & 1u, err);
      tc_fence_after();
      const uint32_t aS = smem_u32(sS), bK = smem_u32(sK + st * AT_SUBTILE);
#pragma unroll
      for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdQ, kmaj(aS, kk), mnmaj(bK, kk), idO, (kb > 0 || kk > 0));
      tc_commit(o_done);
    }
    mbar_wait(o_done, (uint32_t)kb & 1u, err);
    tc_fence_after();
    if (tid == 0 && kb + 2 < nsub) {
      mbar_arrive_expect_tx(&kv_full[st], 2 * AT_SUBTILE);
      tma_load_3d(sK + st * AT_SUBTILE, &tm_qkv64, &kv_full[st], C + h * AT_HS, k0 + 2 * AB_SUB, b);
      tma_load_3d(sV + st * AT_SUBTILE, &tm_qkv64, &kv_full[st], 2 * C + h * AT_HS, k0 + 2 * AB_SUB, b);
    }
    // every thread has waited o_done: the dS buffer is free
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  float v[32];
  {
    uint32_t r[32];
    tmem_ld32(tdQ + lanebase + half * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
  }
  if (q < T) store_row32_bf16(dqkv + ((int64_t)b * T + q) * 3 * (int64_t)C + h * AT_HS + half * 32, v, scale);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tm, 256); }
}

// ============================================================ launchers
void launch_attention_fwd_bf16(LaunchCtx& c, bf16* y, float* lse, const bf16* qkv, int B, int T,
                               int C, int NH) {
  if (C / NH != AT_HS) {
    launch_attention_fwd_simt<bf16>(c, y, lse, qkv, B, T, C, NH);
    return;
  }
  CUtensorMap tq, tq64;
  if (!make_tmap_btw(&tq, qkv, B, T, 3 * C) || !make_tmap_btw(&tq64, qkv, B, T, 3 * C, AB_SUB)) {
    c.host_fail = 1;
    return;
  }
  dim3 grid((T + AT_BLK - 1) / AT_BLK, B * NH);
  cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AF_SMEM);
  launch_pdl(c, attn_fwd_tc_kernel, dim3(grid), dim3(AT_THREADS), AF_SMEM, tq, tq64, y, lse, T, C, NH, 1.f / sqrtf((float)AT_HS), c.err);
}

void launch_attention_bwd_bf16(LaunchCtx& c, bf16* dqkv, const bf16* dy, const bf16* y,
                               const bf16* qkv, const float* lse, float* dsum, int B, int T,
                               int C, int NH) {
  if (C / NH != AT_HS) {
    launch_attention_bwd_simt<bf16>(c, dqkv, dy, y, qkv, lse, dsum, B, T, C, NH, nullptr);
    return;
  }
  CUtensorMap tq, td, tq64, td64;
  if (!make_tmap_btw(&tq, qkv, B, T, 3 * C) || !make_tmap_btw(&td, dy, B, T, C) ||
      !make_tmap_btw(&tq64, qkv, B, T, 3 * C, AB_SUB) || !make_tmap_btw(&td64, dy, B, T, C, AB_SUB)) {
    c.host_fail = 1;
    return;
  }
  const int64_t n = (int64_t)B * T * NH;
  launch_pdl(c, attn_bwd_dsum_kernel, dim3((int)std::min<int64_t>((n + 255) / 256, (int64_t)c.num_sms * 16)), dim3(256), 0, dsum, dy, y, B, T, C, NH);
  const float scale = 1.f / sqrtf((float)AT_HS);
  dim3 grid((T + AT_BLK - 1) / AT_BLK, B * NH);
  cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AKV_SMEM);
  launch_pdl(c, attn_bwd_dkv_tc_kernel, dim3(grid), dim3(AT_THREADS), AKV_SMEM, tq, tq64, td64, dqkv, lse, dsum, T, C, NH, scale, c.err);
  cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AQ_SMEM);
  launch_pdl(c, attn_bwd_dq_tc_kernel, dim3(grid), dim3(AT_THREADS), AQ_SMEM, tq, td, tq64, dqkv, lse, dsum, T, C, NH, scale, c.err);
}
