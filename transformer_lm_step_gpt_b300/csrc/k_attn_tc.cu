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
// words of S (rs) and dP (rd):  p = 2^(s*sl2 - lse*log2e),  ds = p (dp - D).
// KEYROW: the row is a key and the columns are queries (dK/dV kernel; lse
// in natural-log units and D per column, from shared memory), else the row
// is a query (dQ kernel; lse2r = lse*log2e and dr per row).  MASK applies
// the causal mask and, for KEYROW, drops columns at or past colmax (only on
// sub-blocks that cross the diagonal or the end of the sequence).
template <bool KEYROW, bool MASK>
__device__ __forceinline__ void bwd_elementwise(const uint32_t* rs, const uint32_t* rd, const float* lsec,
                                                const float* dc, float lse2r, float dr, float sl2,
                                                int col0, int rowpos, uint8_t* prow, uint8_t* srow,
                                                int rx, int c8base, int colmax = 0) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    float lv[8], dv[8];
    if (KEYROW) {
      const float4 a = *reinterpret_cast<const float4*>(lsec + g * 8);
      const float4 b = *reinterpret_cast<const float4*>(lsec + g * 8 + 4);
      const float4 c = *reinterpret_cast<const float4*>(dc + g * 8);
      const float4 d = *reinterpret_cast<const float4*>(dc + g * 8 + 4);
      const float L2E = 1.4426950408889634f;
      lv[0] = a.x * L2E; lv[1] = a.y * L2E; lv[2] = a.z * L2E; lv[3] = a.w * L2E;
      lv[4] = b.x * L2E; lv[5] = b.y * L2E; lv[6] = b.z * L2E; lv[7] = b.w * L2E;
      dv[0] = c.x; dv[1] = c.y; dv[2] = c.z; dv[3] = c.w; dv[4] = d.x; dv[5] = d.y; dv[6] = d.z; dv[7] = d.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; j++) { lv[j] = lse2r; dv[j] = dr; }
    }
    float p[8], ds[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const float pv = ex2_hw(__uint_as_float(rs[g * 8 + j]) * sl2 - lv[j]);
      float dsv = pv * (__uint_as_float(rd[g * 8 + j]) - dv[j]);
      float pk = pv;
      if (MASK) {  // a masked column may hold stale lse / D: select, do not scale
        const int col = col0 + g * 8 + j;
        const bool ok = KEYROW ? (col >= rowpos && col < colmax) : col <= rowpos;
        pk = ok ? pk : 0.f;
        dsv = ok ? dsv : 0.f;
      }
      p[j] = pk;
      ds[j] = dsv;
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

// Column sums of a warp's 32 rows x 32 columns (lane = row, v[j] = column
// j): a reduce-scatter over the lanes (16 + 8 + 4 + 2 + 1 shuffles); lane l
// returns the sum of column l.
__device__ __forceinline__ float warp_colsum32(float* v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; i++) {
      const float send = up ? v[i] : v[i + off];
      const float keep = up ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// 8 warps: warps w and w+4 read the same TMEM lane quarter (w % 4, i.e. the
// same 32 query or key rows) and split the 128 score columns (half = w / 4
// takes columns 64*half .. 64*half+63) and the 64 output head dims
// (32*half .. 32*half+31).
#define AT_THREADS 256

// ============================================================ forward
// One CTA per (128-query block, b*h), keys walked in 64-row sub-blocks;
// two CTAs share an SM.  Warps 0..7 do the online softmax; warp 8 (one
// thread) issues every TMA load and MMA, so no softmax warp stalls on them:
//   S(j) = q k(j)^T into TMEM S[j%2], issued two sub-blocks ahead (as soon
//          as softmax(j-2) has read that buffer);
//   O_blk(j) = P(j) v(j) into TMEM O[j%2] once P(j) is in shared memory;
//          the softmax warps fold it into their register accumulator
//          (online-softmax rescale) during sub-block j+1;
//   k and v stream through three-stage rings, each stage refilled as soon
//          as the MMA that read it has completed.
// Warps w and w+4 exchange their half-row maxima through a double-buffered
// array and a 64-thread named barrier.
// smem: Q | K ring | V ring (64-row tiles) | P0 P1 ([128 x 64]) | row-max exchange [2][2][128] | barriers
#define AF_KV_STAGES 3
#define AF_THREADS (AT_THREADS + 32)
#define AF_SMEM (1024 + AT_TILE + 2 * AF_KV_STAGES * AT_SUBTILE + 2 * AT_TILE + 2048 + 256)

__global__ void __launch_bounds__(AF_THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                       const __grid_constant__ CUtensorMap tm_qkv64, bf16* y, float* lse, int T,
                       int C, int NH, float scale, int* err) {
  pdl_trigger();
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sQ = sm;
  uint8_t* sK = sm + AT_TILE;                    // [AF_KV_STAGES] x [64 x 64]
  uint8_t* sV = sK + AF_KV_STAGES * AT_SUBTILE;  // [AF_KV_STAGES]
  uint8_t* sP = sV + AF_KV_STAGES * AT_SUBTILE;  // 2 x [128 x 64]
  float* red = reinterpret_cast<float*>(sP + 2 * AT_TILE);  // [2 iterations][2 halves][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * AT_TILE + 2048);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                  // [AF_KV_STAGES]
  uint64_t* v_full = k_full + AF_KV_STAGES;     // [AF_KV_STAGES]
  uint64_t* s_done = v_full + AF_KV_STAGES;     // [2]
  uint64_t* o_done = s_done + 2;                // [2]
  // [2]: 8 warp arrivals for sub-block j on p_ready[j % 2] (two barriers, so
  // the softmax warps, which may run a sub-block ahead of the issuer, never
  // complete a barrier's phase twice before the issuer has waited for it)
  uint64_t* p_ready = o_done + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(p_ready + 2);

  const int nqb = gridDim.y;
  const int qb = nqb - 1 - blockIdx.y;  // the grid starts with the longest rows
  const int bh = blockIdx.x, b = bh / NH, h = bh % NH;
  const int q0 = qb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsub = (min(q0 + AT_BLK, T) + AB_SUB - 1) / AB_SUB;  // key sub-blocks up to the last query

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < AF_KV_STAGES; s++) { mbar_init(&k_full[s], 1); mbar_init(&v_full[s], 1); }
    for (int i = 0; i < 2; i++) {
      mbar_init(&s_done[i], 1);
      mbar_init(&o_done[i], 1);
      mbar_init(&p_ready[i], AT_THREADS / 32);
    }
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA + MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
      const uint32_t idO = tc_idesc_bf16(128, 64, false, true);
      auto load_k = [&](int j) {
        const int s = j % AF_KV_STAGES;
        mbar_arrive_expect_tx(&k_full[s], AT_SUBTILE);
        tma_load_3d(sK + s * AT_SUBTILE, &tm_qkv64, &k_full[s], C + h * AT_HS, j * AB_SUB, b);
      };
      auto load_v = [&](int j) {
        const int s = j % AF_KV_STAGES;
        mbar_arrive_expect_tx(&v_full[s], AT_SUBTILE);
        tma_load_3d(sV + s * AT_SUBTILE, &tm_qkv64, &v_full[s], 2 * C + h * AT_HS, j * AB_SUB, b);
      };
      auto issue_s = [&](int j) {  // S(j) into S[j%2]
        const int s = j % AF_KV_STAGES;
        mbar_wait(&k_full[s], (uint32_t)(j / AF_KV_STAGES) & 1u, err);
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ), bK = smem_u32(sK + s * AT_SUBTILE);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tm + (uint32_t)((j & 1) * 64), kmaj(aQ, kk), kmaj(bK, kk), idS, kk > 0);
        tc_commit(&s_done[j & 1]);
      };
      mbar_arrive_expect_tx(q_full, AT_TILE);
      tma_load_3d(sQ, &tm_qkv, q_full, h * AT_HS, q0, b);
      for (int j = 0; j < AF_KV_STAGES && j < nsub; j++) { load_k(j); load_v(j); }
      mbar_wait(q_full, 0, err);
      issue_s(0);
      if (nsub > 1) issue_s(1);
      for (int j = 0; j < nsub; j++) {
        if (j + AF_KV_STAGES < nsub) {  // S(j) has completed: its k stage takes k(j+3)
          mbar_wait(&s_done[j & 1], (uint32_t)(j >> 1) & 1u, err);
          load_k(j + AF_KV_STAGES);
        }
        mbar_wait(&p_ready[j & 1], (uint32_t)(j >> 1) & 1u, err);  // P(j) written, S[j%2] read
        tc_fence_after();
        {
          const int s = j % AF_KV_STAGES;
          mbar_wait(&v_full[s], (uint32_t)(j / AF_KV_STAGES) & 1u, err);
          tc_fence_after();
          const uint32_t aP = smem_u32(sP + (j & 1) * AT_TILE), bV = smem_u32(sV + s * AT_SUBTILE);
#pragma unroll
          for (int kk = 0; kk < 4; kk++)
            tc_mma_bf16(tm + 128 + (uint32_t)((j & 1) * 64), kmaj(aP, kk), mnmaj(bV, kk), idO, kk > 0);
          tc_commit(&o_done[j & 1]);
        }
        if (j + 2 < nsub) issue_s(j + 2);
        if (j >= 1 && j + 2 < nsub && j + 2 >= AF_KV_STAGES) {  // PV(j-1) has completed: v(j+2)
          mbar_wait(&o_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, err);
          load_v(j + 2);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane, q = q0 + row;
    const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;
    const float sl2 = scale * 1.4426950408889634f;  // scores -> log2 units
    float m = -INFINITY, lpart = 0.f, alpha_prev = 1.f;
    float o[32];
#pragma unroll
    for (int i = 0; i < 32; i++) o[i] = 0.f;

    for (int j = 0; j < nsub; j++) {
      const int sb = j & 1;
      const uint32_t tS = tm + (uint32_t)(sb * 64);
      mbar_wait(&s_done[sb], (uint32_t)(j >> 1) & 1u, err);
      tc_fence_after();
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
      uint8_t* prow = sP + sb * AT_TILE + row * 128;
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
      if (lane == 0) mbar_arrive(&p_ready[sb]);
      // fold in O_blk(j-1) (its MMA ran during this sub-block's softmax); once
      // read, O[(j-1)%2] and P[(j-1)%2] may be reused by PV(j+1) and P(j+1)
      if (j > 0) {
        const int pb = sb ^ 1;
        mbar_wait(&o_done[pb], (uint32_t)((j - 1) >> 1) & 1u, err);
        tc_fence_after();
        uint32_t ro[32];
        tmem_ld32(tm + 128 + (uint32_t)(pb * 64) + lanebase + half * 32, ro);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i++) o[i] = o[i] * alpha_prev + __uint_as_float(ro[i]);
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
    named_bar_sync(5, AT_THREADS);  // every softmax warp is past its last exchange
    red[half * 128 + row] = lpart;
    named_bar_sync(5, AT_THREADS);
    const float l = red[row] + red[128 + row];
    if (q < T) {
      store_row32_bf16(y + ((int64_t)b * T + q) * C + h * AT_HS + half * 32, o, 1.f / l);
      if (half == 0) lse[(int64_t)bh * T + q] = m * scale + logf(l);
    }
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
// One CTA per (128-key block, b*h), queries walked in 64-row sub-blocks,
// warp-specialised so the tensor core never waits for the elementwise work:
//   warp 9      loader: TMA of q and dy sub-blocks into a DKV_STAGES-deep
//               ring, with each sub-block's lse and D (bulk copies on the
//               same barrier when T is a multiple of 4; otherwise all of the
//               block's lse / D are read once, before the first sub-block)
//   warp 8      MMA issuer: S^T(j) = K q(j)^T and dP^T(j) = V dy(j)^T into
//               TMEM buffer j%2, then dV += P^T(j-1) dy(j-1), dK += dS^T(j-1)
//               q(j-1) -- so sub-block j's scores are computed while the
//               compute warps work on j-1
//   warps 0..7  compute: P^T = 2^(S^T*scale*log2e - lse*log2e), dS^T = P^T
//               (dP^T - D) into shared-memory buffer j%2 (two per TMEM lane
//               quarter, splitting the 64 query columns)
// A q / dy stage is refilled only once dV, dK of its sub-block are done, so
// the ring is deep enough to cover that round trip plus the TMA latency.
// TMEM: [S^T | dP^T] x 2 buffers, dV, dK (384 of 512 columns).
// smem: K | V | DKV_STAGES x (q, dy) | 2 x (P^T, dS^T) | barriers | lse / D
// (per stage: [DKV_STAGES][lse 64, D 64]; whole block: lse[Tq], D[Tq] with
// Tq = T - k0 rounded up to 64).  The grid's y index is the key block, so
// the hardware starts the longest blocks (most queries) first.
#define DKV_STAGES 6
#define DKV_THREADS (AT_THREADS + 64)
#define AKV_FIXED (1024 + 2 * AT_TILE + DKV_STAGES * 2 * AT_SUBTILE + 4 * AT_TILE + 256)
static inline bool akv_staged_ld(int T) { return T % 4 == 0; }
static inline size_t akv_smem(int T) {
  const size_t whole = 8 * (size_t)((T + 63) / 64 * 64);
  return AKV_FIXED + (akv_staged_ld(T) ? (size_t)DKV_STAGES * 512 : whole);
}

__global__ void __launch_bounds__(DKV_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_qkv64,
                           const __grid_constant__ CUtensorMap tm_dy64, bf16* dqkv, const float* lse,
                           const float* dsum, float* bias_partial, int T, int C, int NH, float scale,
                           int* err) {
  pdl_trigger();
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sK = sm;
  uint8_t* sV = sm + AT_TILE;
  uint8_t* sQ = sm + 2 * AT_TILE;                     // [DKV_STAGES] x [64 x 64]
  uint8_t* sD = sQ + DKV_STAGES * AT_SUBTILE;         // dy, [DKV_STAGES]
  uint8_t* sP = sD + DKV_STAGES * AT_SUBTILE;         // P^T  [2] x [128 keys x 64 queries]
  uint8_t* sS = sP + 2 * AT_TILE;                     // dS^T [2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + 2 * AT_TILE);
  uint64_t* kv_full = bars;
  uint64_t* ld_full = bars + 1;                  // whole-block lse / D written
  uint64_t* q_full = bars + 2;                   // [DKV_STAGES]: TMA bytes
  uint64_t* q_empty = q_full + DKV_STAGES;       // [DKV_STAGES]: MMA commit
  uint64_t* s_full = q_empty + DKV_STAGES;       // [2]: S^T, dP^T ready
  uint64_t* s_empty = s_full + 2;                // [2]: compute warps have read them
  uint64_t* p_full = s_empty + 2;                // [2]: P^T, dS^T written
  uint64_t* p_empty = p_full + 2;                // [2]: dV/dK MMAs have read them
  uint64_t* done = p_empty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  float* sLD = reinterpret_cast<float*>(sS + 2 * AT_TILE + 256);
  const int kb = blockIdx.y;  // key block
  const int bh = blockIdx.x, b = bh / NH, h = bh % NH;
  const int k0 = kb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsub = (T - k0 + AB_SUB - 1) / AB_SUB;  // 64-query sub-blocks from k0 to T
  const bool staged = (T & 3) == 0;                 // per-stage lse / D bulk copies

  if (tid == 0) {
    mbar_init(kv_full, 1);
    mbar_init(ld_full, 1);
    for (int s = 0; s < DKV_STAGES; s++) { mbar_init(&q_full[s], 1); mbar_init(&q_empty[s], 1); }
    for (int i = 0; i < 2; i++) {
      mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 8);
      mbar_init(&p_full[i], 8); mbar_init(&p_empty[i], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_qkv64);
    tma_prefetch_desc(&tm_dy64);
  }
  if (warp == 8) { tmem_alloc(tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_wait();  // from here on global memory written by the previous kernel is read
  const uint32_t tdV = tm + 256, tdK = tm + 320;
  const float sl2 = scale * 1.4426950408889634f;
  const float* lrow = lse + (int64_t)bh * T + k0;
  const float* drow = dsum + (int64_t)bh * T + k0;

  if (warp == 9) {
    // ---------------------------------------------------------------- loader
    auto issue = [&](int j) {
      const int s = j % DKV_STAGES, q0 = k0 + j * AB_SUB;
      const uint32_t ldb = staged ? 4u * (uint32_t)min(AB_SUB, T - q0) : 0u;  // a multiple of 16
      mbar_arrive_expect_tx(&q_full[s], 2 * AT_SUBTILE + 2 * ldb);
      tma_load_3d(sQ + s * AT_SUBTILE, &tm_qkv64, &q_full[s], h * AT_HS, q0, b);
      tma_load_3d(sD + s * AT_SUBTILE, &tm_dy64, &q_full[s], h * AT_HS, q0, b);
      if (staged) {
        bulk_load(sLD + s * 128, lrow + j * AB_SUB, ldb, &q_full[s]);
        bulk_load(sLD + s * 128 + 64, drow + j * AB_SUB, ldb, &q_full[s]);
      }
    };
    int j = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * AT_TILE);
      tma_load_3d(sK, &tm_qkv, kv_full, C + h * AT_HS, k0, b);
      tma_load_3d(sV, &tm_qkv, kv_full, 2 * C + h * AT_HS, k0, b);
      for (; j < nsub && j < DKV_STAGES; j++) issue(j);
    }
    if (!staged) {
      float* sL = sLD;
      float* sDd = sLD + nsub * AB_SUB;
      const int nq = nsub * AB_SUB;
      for (int i0 = 0; i0 < nq; i0 += 32 * 16) {  // 32 loads in flight per lane
        float lv[16], dv[16];
#pragma unroll
        for (int u = 0; u < 16; u++) {
          const int i = i0 + u * 32 + lane;
          const bool in = i < nq && k0 + i < T;
          lv[u] = in ? __ldg(lrow + i) : 0.f;
          dv[u] = in ? __ldg(drow + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; u++) {
          const int i = i0 + u * 32 + lane;
          if (i < nq) { sL[i] = lv[u]; sDd[i] = dv[u]; }
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(ld_full);
      for (j = DKV_STAGES; j < nsub; j++) {
        mbar_wait(&q_empty[j % DKV_STAGES], ((uint32_t)(j / DKV_STAGES) & 1u) ^ 1u, err);
        issue(j);
      }
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
      const uint32_t idO = tc_idesc_bf16(128, 64, false, true);
      mbar_wait(kv_full, 0, err);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      for (int j = 0; j <= nsub; j++) {
        if (j < nsub) {
          const int s = j % DKV_STAGES, bf = j & 1;
          mbar_wait(&q_full[s], (uint32_t)(j / DKV_STAGES) & 1u, err);
          mbar_wait(&s_empty[bf], ((uint32_t)(j >> 1) & 1u) ^ 1u, err);
          tc_fence_after();
          const uint32_t bQ = smem_u32(sQ + s * AT_SUBTILE), bD = smem_u32(sD + s * AT_SUBTILE);
          const uint32_t tS = tm + (uint32_t)(bf * 128), tP = tS + 64;
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tS, kmaj(aK, kk), kmaj(bQ, kk), idS, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tP, kmaj(aV, kk), kmaj(bD, kk), idS, kk > 0);
          tc_commit(&s_full[bf]);
        }
        if (j >= 1) {
          const int jj = j - 1, s = jj % DKV_STAGES, bf = jj & 1;
          mbar_wait(&p_full[bf], (uint32_t)(jj >> 1) & 1u, err);
          tc_fence_after();
          const uint32_t aP = smem_u32(sP + bf * AT_TILE), aS = smem_u32(sS + bf * AT_TILE);
          const uint32_t bQ = smem_u32(sQ + s * AT_SUBTILE), bD = smem_u32(sD + s * AT_SUBTILE);
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdV, kmaj(aP, kk), mnmaj(bD, kk), idO, (jj > 0 || kk > 0));
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdK, kmaj(aS, kk), mnmaj(bQ, kk), idO, (jj > 0 || kk > 0));
          tc_commit(&p_empty[bf]);
          tc_commit(&q_empty[s]);
        }
      }
      tc_commit(done);
    }
  } else {
    // ---------------------------------------------------------------- compute warps
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane, key = k0 + row;
    const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;
    mbar_wait(ld_full, 0, err);
    for (int j = 0; j < nsub; j++) {
      const int bf = j & 1, s = j % DKV_STAGES;
      const int q0 = k0 + j * AB_SUB;
      mbar_wait(&s_full[bf], (uint32_t)(j >> 1) & 1u, err);
      tc_fence_after();
      uint32_t rs[32], rd[32];
      const uint32_t tS = tm + (uint32_t)(bf * 128);
      tmem_ld32(tS + lanebase + half * 32, rs);
      tmem_ld32(tS + 64 + lanebase + half * 32, rd);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[bf]);
      mbar_wait(&p_empty[bf], ((uint32_t)(j >> 1) & 1u) ^ 1u, err);  // P^T / dS^T buffer free
      if (staged) mbar_wait(&q_full[s], (uint32_t)(j / DKV_STAGES) & 1u, err);  // the stage's lse / D
      const float* lc = staged ? sLD + s * 128 + half * 32 : sLD + j * AB_SUB + half * 32;
      const float* dc = staged ? sLD + s * 128 + 64 + half * 32 : sLD + (nsub + j) * AB_SUB + half * 32;
      uint8_t* prow = sP + bf * AT_TILE + row * 128;
      uint8_t* srow = sS + bf * AT_TILE + row * 128;
      if (q0 < k0 + AT_BLK || q0 + AB_SUB > T)
        bwd_elementwise<true, true>(rs, rd, lc, dc, 0.f, 0.f, sl2, q0 + half * 32, key, prow, srow,
                                    row & 7, half * 4, T);
      else
        bwd_elementwise<true, false>(rs, rd, lc, dc, 0.f, 0.f, sl2, q0 + half * 32, key, prow, srow,
                                     row & 7, half * 4);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[bf]);
    }
    mbar_wait(done, 0, err);
    tc_fence_after();
    const int64_t C3 = 3 * (int64_t)C;
    float* red = reinterpret_cast<float*>(sP);  // [2][4][64]: free once every MMA is done
    float v[32];
    uint32_t r[32];
    tmem_ld32(tdV + lanebase + half * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = key < T ? __uint_as_float(r[i]) : 0.f;
    if (key < T) store_row32_bf16(dqkv + ((int64_t)b * T + key) * C3 + 2 * C + h * AT_HS + half * 32, v, 1.f);
    red[quarter * 64 + half * 32 + lane] = warp_colsum32(v);
    tmem_ld32(tdK + lanebase + half * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = key < T ? __uint_as_float(r[i]) : 0.f;
    if (key < T) store_row32_bf16(dqkv + ((int64_t)b * T + key) * C3 + C + h * AT_HS + half * 32, v, scale);
    red[256 + quarter * 64 + half * 32 + lane] = warp_colsum32(v) * scale;
    // the block's column sums of dV and dK: one partial row of the qkv bias
    // gradient per (batch row, key block)
    named_bar_sync(1, AT_THREADS);
    if (tid < 128) {
      const int which = tid >> 6, col = tid & 63;  // 0: dV, 1: dK
      const float* rr = red + which * 256 + col;
      const float sum = (rr[0] + rr[64]) + (rr[128] + rr[192]);
      bias_partial[((int64_t)b * gridDim.y + kb) * C3 + (which ? C : 2 * C) + h * AT_HS + col] = sum;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) { tc_fence_after(); tmem_dealloc(tm, 512); }
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
                          const float* dsum, float* bias_partial, int T, int C, int NH, float scale,
                          int* err) {
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

  const int nqb = gridDim.y;
  const int qb = nqb - 1 - blockIdx.y;  // the grid starts with the blocks that meet the most keys
  const int bh = blockIdx.x, b = bh / NH, h = bh % NH;
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
    for (int j = 0; j < 32; j++) v[j] = q < T ? __uint_as_float(r[j]) : 0.f;
  }
  if (q < T) store_row32_bf16(dqkv + ((int64_t)b * T + q) * 3 * (int64_t)C + h * AT_HS + half * 32, v, scale);
  // the block's column sums of dQ: one partial row of the qkv bias gradient
  // per (batch row, query block); the dS buffer is free after the loop
  float* red = reinterpret_cast<float*>(sS);  // [4][64]
  red[quarter * 64 + half * 32 + lane] = warp_colsum32(v) * scale;
  __syncthreads();
  if (tid < 64) {
    const float* rr = red + tid;
    bias_partial[((int64_t)b * nqb + qb) * 3 * (int64_t)C + h * AT_HS + tid] = (rr[0] + rr[64]) + (rr[128] + rr[192]);
  }
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
  dim3 grid(B * NH, (T + AT_BLK - 1) / AT_BLK);
  cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AF_SMEM);
  launch_pdl(c, attn_fwd_tc_kernel, dim3(grid), dim3(AF_THREADS), AF_SMEM, tq, tq64, y, lse, T, C, NH, 1.f / sqrtf((float)AT_HS), c.err);
}

bool launch_attention_bwd_bf16(LaunchCtx& c, bf16* dqkv, const bf16* dy, const bf16* y,
                               const bf16* qkv, const float* lse, float* dsum, int B, int T,
                               int C, int NH, float* bias_partial) {
  if (C / NH != AT_HS) {
    launch_attention_bwd_simt<bf16>(c, dqkv, dy, y, qkv, lse, dsum, B, T, C, NH, nullptr);
    return false;
  }
  CUtensorMap tq, td, tq64, td64;
  if (!make_tmap_btw(&tq, qkv, B, T, 3 * C) || !make_tmap_btw(&td, dy, B, T, C) ||
      !make_tmap_btw(&tq64, qkv, B, T, 3 * C, AB_SUB) || !make_tmap_btw(&td64, dy, B, T, C, AB_SUB)) {
    c.host_fail = 1;
    return false;
  }
  const int64_t n = (int64_t)B * T * NH;
  launch_pdl(c, attn_bwd_dsum_kernel, dim3((int)std::min<int64_t>((n + 255) / 256, (int64_t)c.num_sms * 16)), dim3(256), 0, dsum, dy, y, B, T, C, NH);
  const float scale = 1.f / sqrtf((float)AT_HS);
  dim3 grid(B * NH, (T + AT_BLK - 1) / AT_BLK);
  const size_t kv_smem = akv_smem(T);
  cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kv_smem);
  launch_pdl(c, attn_bwd_dkv_tc_kernel, dim3(grid), dim3(DKV_THREADS), kv_smem, tq, tq64, td64, dqkv, lse, dsum, bias_partial, T, C, NH, scale, c.err);
  cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AQ_SMEM);
  launch_pdl(c, attn_bwd_dq_tc_kernel, dim3(grid), dim3(AT_THREADS), AQ_SMEM, tq, td, tq64, dqkv, lse, dsum, bias_partial, T, C, NH, scale, c.err);
  return true;
}
