// k_attn_tc.cu -- causal multi-head self-attention on the tcgen05 tensor cores.
//
// GeekNews, "A GPT-2-based ChatGPT clone in 3000 bytes of C", section "The
// Transformer core": per head, S = q k^T (scaled by 1/sqrt(hs)), the lower-
// triangular causal mask, softmax over each query row, times v.  Here the
// T x T score matrix is never stored: it is computed one 128 x 128 tile at a
// time in TMEM and folded into an online softmax (forward) or recomputed from
// the saved row logsumexp (backward).
//
// Head size 64.  Every tile of q, k, v, dy is one TMA box [128 or 64 rows x
// 64] of a 3-D tensor map over [B, T, width] (rows past T read as zero),
// landing 128-byte-swizzled in shared memory, where a tcgen05 descriptor can
// read it either as a K-major operand (rows = M or N) or as an MN-major one
// (rows = K) -- so S = q k^T, P v, dV = P^T dy, dK = dS^T q and dQ = dS k all
// read the same tiles.  Each kernel is warp-specialised: one thread issues
// the TMA loads and MMAs, the other warps do the elementwise work, and every
// hand-off is an mbarrier.
//
//   forward   one CTA per (128-query block, b*h), 64-key sub-blocks: S -> TMEM
//             (two buffers, issued two sub-blocks ahead), online softmax by 8
//             warps (thread = query row), P -> smem, O += P v accumulated in
//             TMEM; the softmax reference maximum moves only when a row's
//             maximum grows by more than 2^8, and only then is O rescaled in
//             place.  Saves lse in base 2: max*scale*log2e + log2(sum).
//   backward  D = rowsum(dy * y); one CTA per (128-key block, b*h) for dK, dV
//             over 128-query sub-blocks (S^T, dP^T recomputed into TMEM; P^T
//             and dS^T written back to TMEM and read there as the A operand
//             of dV += P^T dy, dK += dS^T q); one CTA per (128-query block,
//             b*h) for dQ over 64-key sub-blocks (dQ += dS k, dS in smem).
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
static bool make_tmap_btw(CUtensorMap* m, const void* base, int B, int T, int W, int rows = 128);
bool attn_tmap_btw(CUtensorMap* m, const void* base, int B, int T, int W, int rows) {
  return make_tmap_btw(m, base, B, T, W, rows);
}
static bool make_tmap_btw(CUtensorMap* m, const void* base, int B, int T, int W, int rows) {
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
// Write 8 consecutive bf16 values (16-byte chunk c8 of a row) into a
// 128B-swizzled [rows x 64] buffer (one atom), given the row's base pointer
// (buf + r*128) and its swizzle (r & 7).
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

// The dQ kernel's elementwise step for 32 key columns of one query row,
// from the TMEM words of S (rs) and dP (rd): p = 2^(s*sl2 - lse2), ds =
// p (dp - D), with the row's lse2 (base-2 units, as the forward saves it)
// and D; dS (bf16) goes to the row's 16-byte chunks c8base.. of a
// 128B-swizzled [rows x 64] atom (srow = atom + r*128, rx = r & 7).  MASK
// applies the causal mask (only on sub-blocks that cross the diagonal).
template <bool MASK>
__device__ __forceinline__ void qrow_elementwise(const uint32_t* rs, const uint32_t* rd, float lse2r, float dr,
                                                 float sl2, int col0, int rowpos, uint8_t* srow, int rx,
                                                 int c8base) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    float ds[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const float pv = ex2_hw(__uint_as_float(rs[g * 8 + j]) * sl2 - lse2r);
      float dsv = pv * (__uint_as_float(rd[g * 8 + j]) - dr);
      if (MASK) dsv = col0 + g * 8 + j <= rowpos ? dsv : 0.f;
      ds[j] = dsv;
    }
    st_row8(srow, rx, c8base + g, ds);
  }
}

// The dK/dV kernel's elementwise step for 32 query columns of one key row,
// kept in registers: P^T and dS^T as packed bf16 pairs (pk, dk: 16 words
// each, column pairs in order), so they can be computed before the shared-
// memory buffer they go to is free.  lse2c: the columns' lse in base-2
// units (as the forward saves it), dc: their D, both from shared memory.
template <bool MASK>
__device__ __forceinline__ void keyrow_pack(const uint32_t* rs, const uint32_t* rd, const float* lse2c,
                                            const float* dc, float sl2, int col0, int key, int colmax,
                                            uint32_t* pk, uint32_t* dk) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    const float4 a = *reinterpret_cast<const float4*>(lse2c + g * 8);
    const float4 bq = *reinterpret_cast<const float4*>(lse2c + g * 8 + 4);
    const float4 c = *reinterpret_cast<const float4*>(dc + g * 8);
    const float4 d = *reinterpret_cast<const float4*>(dc + g * 8 + 4);
    const float lv[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
    const float dv[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
    float p[8], ds[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const float pv = ex2_hw(__uint_as_float(rs[g * 8 + j]) * sl2 - lv[j]);
      float dsv = pv * (__uint_as_float(rd[g * 8 + j]) - dv[j]);
      float pkv = pv;
      if (MASK) {  // a masked column may hold stale lse / D: select, do not scale
        const int col = col0 + g * 8 + j;
        const bool ok = col >= key && col < colmax;
        pkv = ok ? pkv : 0.f;
        dsv = ok ? dsv : 0.f;
      }
      p[j] = pkv;
      ds[j] = dsv;
    }
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      __nv_bfloat162 tp = __floats2bfloat162_rn(p[j], p[j + 1]);
      __nv_bfloat162 td = __floats2bfloat162_rn(ds[j], ds[j + 1]);
      pk[g * 4 + j / 2] = *reinterpret_cast<uint32_t*>(&tp);
      dk[g * 4 + j / 2] = *reinterpret_cast<uint32_t*>(&td);
    }
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
// thread) issues every MMA and warp 9 (one thread) every TMA load, so no
// softmax warp stalls on them and no load waits behind an MMA hand-off:
//   S(j) = q k(j)^T into TMEM S[j%2], issued two sub-blocks ahead (as soon
//          as softmax(j-2) has read that buffer);
//   O += P(j) v(j) into one TMEM accumulator once P(j) is in shared
//          memory; the softmax warps take P relative to a reference maximum
//          that moves only when a row's maximum exceeds it by more than 8 in
//          log2 units (P <= 2^8), and then rescale O in TMEM after PV(j-1)
//          has completed and before they release P(j) (lazy rescaling);
//   k and v stream through three-stage rings, each stage refilled by the
//          loader as soon as the MMA that read it has completed (k_empty /
//          v_empty, committed with the MMAs).
// Warps w and w+4 exchange their half-row maxima through a double-buffered
// array and a 64-thread named barrier.
// TMEM: S0 S1 (columns 0..127), O (128..191).
// smem: Q | K ring | V ring (64-row tiles) | P0 P1 ([128 x 64]) | row-max exchange [2][2][128] | barriers
#define AF_KV_STAGES 3
#define AF_THREADS (AT_THREADS + 64)
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
  uint64_t* k_empty = p_ready + 2;               // [AF_KV_STAGES]: S of the stage done
  uint64_t* v_empty = k_empty + AF_KV_STAGES;    // [AF_KV_STAGES]: PV of the stage done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(v_empty + AF_KV_STAGES);

  const int nqb = gridDim.y;
  const int qb = nqb - 1 - blockIdx.y;  // the grid starts with the longest rows
  const int bh = blockIdx.x, b = bh / NH, h = bh % NH;
  const int q0 = qb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsub = (min(q0 + AT_BLK, T) + AB_SUB - 1) / AB_SUB;  // key sub-blocks up to the last query

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < AF_KV_STAGES; s++) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
      const uint32_t idO = tc_idesc_bf16(128, 64, false, true);
      auto issue_s = [&](int j) {  // S(j) into S[j%2]; its k stage is then free
        const int s = j % AF_KV_STAGES;
        mbar_wait(&k_full[s], (uint32_t)(j / AF_KV_STAGES) & 1u, err);
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ), bK = smem_u32(sK + s * AT_SUBTILE);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tm + (uint32_t)((j & 1) * 64), kmaj(aQ, kk), kmaj(bK, kk), idS, kk > 0);
        tc_commit(&s_done[j & 1]);
        tc_commit(&k_empty[s]);
      };
      mbar_wait(q_full, 0, err);
      issue_s(0);
      if (nsub > 1) issue_s(1);
      for (int j = 0; j < nsub; j++) {
        mbar_wait(&p_ready[j & 1], (uint32_t)(j >> 1) & 1u, err);  // P(j) written, S[j%2] read
        tc_fence_after();
        const int s = j % AF_KV_STAGES;
        mbar_wait(&v_full[s], (uint32_t)(j / AF_KV_STAGES) & 1u, err);
        tc_fence_after();
        const uint32_t aP = smem_u32(sP + (j & 1) * AT_TILE), bV = smem_u32(sV + s * AT_SUBTILE);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tm + 128, kmaj(aP, kk), mnmaj(bV, kk), idO, (j > 0 || kk > 0));
        tc_commit(&o_done[j & 1]);
        tc_commit(&v_empty[s]);
        if (j + 2 < nsub) issue_s(j + 2);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ TMA loader
    // q once; k(j) and v(j) into their ring stages as soon as the MMA that
    // read the stage's previous tile (S(j-3), PV(j-3)) has completed
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, AT_TILE);
      tma_load_3d(sQ, &tm_qkv, q_full, h * AT_HS, q0, b);
      for (int j = 0; j < nsub; j++) {
        const int s = j % AF_KV_STAGES;
        const uint32_t ph = (uint32_t)(j / AF_KV_STAGES - 1) & 1u;
        if (j >= AF_KV_STAGES) mbar_wait(&k_empty[s], ph, err);
        mbar_arrive_expect_tx(&k_full[s], AT_SUBTILE);
        tma_load_3d(sK + s * AT_SUBTILE, &tm_qkv64, &k_full[s], C + h * AT_HS, j * AB_SUB, b);
        if (j >= AF_KV_STAGES) mbar_wait(&v_empty[s], ph, err);
        mbar_arrive_expect_tx(&v_full[s], AT_SUBTILE);
        tma_load_3d(sV + s * AT_SUBTILE, &tm_qkv64, &v_full[s], 2 * C + h * AT_HS, j * AB_SUB, b);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane, q = q0 + row;
    const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;
    const float sl2 = scale * 1.4426950408889634f;  // scores -> log2 units
    // m: the row's reference maximum (raw score units).  P and the row sum
    // are taken relative to it; it moves only when a new maximum exceeds it
    // by more than 8 in log2 units (so P <= 2^8), and then the accumulator O
    // in TMEM and the row sum are rescaled by 2^((m_old - m_new) * sl2).
    float m = -INFINITY, lpart = 0.f;

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
      const float mcand = fmaxf(m, fmaxf(rd[row], rd[128 + row]));
      const bool resc = (mcand - m) * sl2 > 8.f;  // always at j = 0 (m = -inf)
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_hw((m - mcand) * sl2);
        lpart *= alpha;
        m = mcand;
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        // O holds PV(0 .. j-1) once PV(j-1) completes; PV(j) waits for this
        // sub-block's p_ready, so the rescale cannot race an MMA
        mbar_wait(&o_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, err);
        tc_fence_after();
        const uint32_t tO = tm + 128 + lanebase + half * 32;
        uint32_t ro[32];
        tmem_ld32(tO, ro);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i++) ro[i] = __float_as_uint(__uint_as_float(ro[i]) * alpha);
        tmem_st16(tO, ro);
        tmem_st16(tO + 16, ro + 16);
        tmem_st_wait();
      }
      // P[sb] was read by PV(j-2)
      if (j >= 2) mbar_wait(&o_done[sb], (uint32_t)((j - 2) >> 1) & 1u, err);
      const float mo = m * sl2;
      // pass 2: P = 2^(scale (s - m) log2 e) -> smem P[sb] (bf16), partial row sum
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
      lpart += sum;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[sb]);
    }
    float o[32];
    {  // O = PV(0 .. nsub-1), relative to the final reference maximum
      const int pb = (nsub - 1) & 1;
      mbar_wait(&o_done[pb], (uint32_t)((nsub - 1) >> 1) & 1u, err);
      tc_fence_after();
      uint32_t ro[32];
      tmem_ld32(tm + 128 + lanebase + half * 32, ro);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; i++) o[i] = __uint_as_float(ro[i]);
    }
    named_bar_sync(5, AT_THREADS);  // every softmax warp is past its last exchange
    red[half * 128 + row] = lpart;
    named_bar_sync(5, AT_THREADS);
    const float l = red[row] + red[128 + row];
    if (q < T) {
      store_row32_bf16(y + ((int64_t)b * T + q) * C + h * AT_HS + half * 32, o, 1.f / l);
      if (half == 0) lse[(int64_t)bh * T + q] = m * sl2 + log2f(l);  // base-2 units
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
// One CTA per (128-key block, b*h), queries walked in 128-row sub-blocks,
// warp-specialised:
//   warp 9      loader: TMA of the q and dy tiles into a DKV_STAGES-deep
//               ring, with each sub-block's lse and D (bulk copies on the
//               same barrier when T is a multiple of 4; otherwise all of the
//               block's lse / D are read once, before the first sub-block)
//   warp 16     MMA issuer: S^T(j) = K q(j)^T and dP^T(j) = V dy(j)^T
//               (N = 128) into TMEM, then dV += P^T(j-1) dy(j-1) and dK +=
//               dS^T(j-1) q(j-1) (N = 64, K = 128 queries) with P^T and dS^T
//               read from TMEM (the A operand), dy and q from shared memory
//   warps 0..15 compute: copy S^T(j), dP^T(j) to registers at once (so
//               S^T(j+1) runs during their elementwise work), then P^T =
//               2^(S^T*scale*log2e - lse2), dS^T = P^T (dP^T - D) as
//               packed bf16 into TMEM (warps w, w+4, w+8, w+12 share TMEM
//               lane quarter w%4 and take 32 of the 128 query columns each;
//               the math runs before the buffer wait, so it overlaps
//               dV/dK(j-1))
// Keeping P^T and dS^T out of shared memory saves their stores and the
// MMAs' shared-memory operand reads (an M = 128, N = 64, K = 16 MMA takes
// about 75 cycles whether A comes from tensor or shared memory).
// A q / dy stage is refilled once dV, dK of its sub-block are done.
// TMEM: S^T 0..127, dP^T 128..255, dV 256..319, dK 320..383, P^T 384..447,
// dS^T 448..511 (bf16 pairs).
// smem: K | V | DKV_STAGES x (q, dy) | barriers | lse / D
// (per stage: [DKV_STAGES][lse 128, D 128]; whole block: lse[Tq], D[Tq] with
// Tq = T - k0 rounded up to 128).  The grid's y index is the key block, so
// the hardware starts the longest blocks (most queries) first.
#define DKV_SUB 128
#define DKV_STAGES 4
#define DKV_CWARPS 16
#define DKV_THREADS (DKV_CWARPS * 32 + 64)
#define AKV_FIXED (1024 + 2 * AT_TILE + DKV_STAGES * 2 * AT_TILE + 256)
static inline size_t akv_smem(int T) {
  const size_t whole = 8 * (size_t)((T + DKV_SUB - 1) / DKV_SUB * DKV_SUB);
  return AKV_FIXED + ((T % 4 == 0) ? (size_t)DKV_STAGES * 8 * DKV_SUB : whole);
}

__global__ void __launch_bounds__(DKV_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_dy, bf16* dqkv, const float* lse,
                           const float* dsum, float* bias_partial, int T, int C, int NH, float scale,
                           int* err) {
  pdl_trigger();
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sK = sm;
  uint8_t* sV = sm + AT_TILE;
  uint8_t* sQ = sm + 2 * AT_TILE;                // [DKV_STAGES] x [128 x 64]
  uint8_t* sD = sQ + DKV_STAGES * AT_TILE;       // dy, [DKV_STAGES]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sD + DKV_STAGES * AT_TILE);
  uint64_t* kv_full = bars;
  uint64_t* ld_full = bars + 1;                  // whole-block lse / D written
  uint64_t* q_full = bars + 2;                   // [DKV_STAGES]: TMA bytes
  uint64_t* q_empty = q_full + DKV_STAGES;       // [DKV_STAGES]: dV, dK of the stage done
  uint64_t* s_full = q_empty + DKV_STAGES;       // S^T, dP^T in TMEM
  uint64_t* s_empty = s_full + 1;                // 8 warps have copied them out
  uint64_t* p_full = s_empty + 1;                // 8 warps have written P^T, dS^T
  uint64_t* p_empty = p_full + 1;                // dV, dK MMAs have read them
  uint64_t* done = p_empty + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  float* sLD = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);
  const int kb = blockIdx.y;  // key block
  const int bh = blockIdx.x, b = bh / NH, h = bh % NH;
  const int k0 = kb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsub = (T - k0 + DKV_SUB - 1) / DKV_SUB;  // 128-query sub-blocks from k0 to T
  const bool staged = (T & 3) == 0;                   // per-stage lse / D bulk copies

  if (tid == 0) {
    mbar_init(kv_full, 1);
    mbar_init(ld_full, 1);
    for (int s = 0; s < DKV_STAGES; s++) { mbar_init(&q_full[s], 1); mbar_init(&q_empty[s], 1); }
    mbar_init(s_full, 1);
    mbar_init(s_empty, DKV_CWARPS);
    mbar_init(p_full, DKV_CWARPS);
    mbar_init(p_empty, 1);
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_dy);
  }
  if (warp == DKV_CWARPS) { tmem_alloc(tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_wait();  // from here on global memory written by the previous kernel is read
  const uint32_t tSt = tm, tdPt = tm + 128, tdV = tm + 256, tdK = tm + 320, tPt = tm + 384, tdSt = tm + 448;
  const float sl2 = scale * 1.4426950408889634f;
  const float* lrow = lse + (int64_t)bh * T + k0;
  const float* drow = dsum + (int64_t)bh * T + k0;

  if (warp == DKV_CWARPS + 1) {
    // ---------------------------------------------------------------- loader
    auto issue = [&](int j) {
      const int s = j % DKV_STAGES, q0 = k0 + j * DKV_SUB;
      const uint32_t ldb = staged ? 4u * (uint32_t)min(DKV_SUB, T - q0) : 0u;  // a multiple of 16
      mbar_arrive_expect_tx(&q_full[s], 2 * AT_TILE + 2 * ldb);
      tma_load_3d(sQ + s * AT_TILE, &tm_qkv, &q_full[s], h * AT_HS, q0, b);
      tma_load_3d(sD + s * AT_TILE, &tm_dy, &q_full[s], h * AT_HS, q0, b);
      if (staged) {
        bulk_load(sLD + s * 2 * DKV_SUB, lrow + j * DKV_SUB, ldb, &q_full[s]);
        bulk_load(sLD + s * 2 * DKV_SUB + DKV_SUB, drow + j * DKV_SUB, ldb, &q_full[s]);
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
      float* sDd = sLD + nsub * DKV_SUB;
      const int nq = nsub * DKV_SUB;
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
  } else if (warp == DKV_CWARPS) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 128, false, false);
      const uint32_t idO = tc_idesc_bf16(128, 64, false, true);
      mbar_wait(kv_full, 0, err);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      for (int j = 0; j <= nsub; j++) {
        if (j < nsub) {
          const int s = j % DKV_STAGES;
          mbar_wait(&q_full[s], (uint32_t)(j / DKV_STAGES) & 1u, err);
          if (j > 0) mbar_wait(s_empty, (uint32_t)(j - 1) & 1u, err);  // S^T(j-1), dP^T(j-1) copied out
          tc_fence_after();
          const uint32_t bQ = smem_u32(sQ + s * AT_TILE), bD = smem_u32(sD + s * AT_TILE);
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tSt, kmaj(aK, kk), kmaj(bQ, kk), idS, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdPt, kmaj(aV, kk), kmaj(bD, kk), idS, kk > 0);
          tc_commit(s_full);
        }
        if (j >= 1) {
          const int jj = j - 1, s = jj % DKV_STAGES;
          mbar_wait(p_full, (uint32_t)jj & 1u, err);
          tc_fence_after();
          const uint32_t bQ = smem_u32(sQ + s * AT_TILE), bD = smem_u32(sD + s * AT_TILE);
#pragma unroll
          for (int kk = 0; kk < 8; kk++) tc_mma_bf16_ts(tdV, tPt + kk * 8, mnmaj(bD, kk), idO, (jj > 0 || kk > 0));
#pragma unroll
          for (int kk = 0; kk < 8; kk++) tc_mma_bf16_ts(tdK, tdSt + kk * 8, mnmaj(bQ, kk), idO, (jj > 0 || kk > 0));
          tc_commit(p_empty);
          tc_commit(&q_empty[s]);
        }
      }
      tc_commit(done);
    }
  } else {
    // ---------------------------------------------------------------- compute warps
    const int quarter = warp & 3, colq = warp >> 2;  // lane quarter, 32-column group
    const int row = quarter * 32 + lane, key = k0 + row;
    const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;
    mbar_wait(ld_full, 0, err);
    for (int j = 0; j < nsub; j++) {
      const int s = j % DKV_STAGES;
      const int q0 = k0 + j * DKV_SUB;
      mbar_wait(s_full, (uint32_t)j & 1u, err);
      tc_fence_after();
      uint32_t rs[32], rd[32];
      tmem_ld32(tSt + lanebase + colq * 32, rs);
      tmem_ld32(tdPt + lanebase + colq * 32, rd);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      if (staged) mbar_wait(&q_full[s], (uint32_t)(j / DKV_STAGES) & 1u, err);  // the stage's lse / D
      const float* lc = (staged ? sLD + s * 2 * DKV_SUB : sLD + j * DKV_SUB) + colq * 32;
      const float* dc = (staged ? sLD + s * 2 * DKV_SUB + DKV_SUB : sLD + (nsub + j) * DKV_SUB) + colq * 32;
      const int c0 = q0 + colq * 32;
      // the math runs while dV, dK(j-1) still read the shared-memory buffers
      uint32_t pk[16], dk[16];
      if (q0 < k0 + AT_BLK || q0 + DKV_SUB > T) keyrow_pack<true>(rs, rd, lc, dc, sl2, c0, key, T, pk, dk);
      else keyrow_pack<false>(rs, rd, lc, dc, sl2, c0, key, T, pk, dk);
      if (j > 0) mbar_wait(p_empty, (uint32_t)(j - 1) & 1u, err);  // dV, dK(j-1) have read P^T, dS^T
      tc_fence_after();
      tmem_st16(tPt + lanebase + colq * 16, pk);
      tmem_st16(tdSt + lanebase + colq * 16, dk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    mbar_wait(done, 0, err);
    tc_fence_after();
    // epilogue: column groups 0, 1 take dV columns 0..31, 32..63; 2, 3 take dK
    const int64_t C3 = 3 * (int64_t)C;
    const int which = colq >> 1, cc = (colq & 1) * 32;  // which: 0 dV, 1 dK
    const float mul = which ? scale : 1.f;
    float* red = reinterpret_cast<float*>(sQ);  // [2][4][64]: the q ring is free once every MMA is done
    float v[32];
    uint32_t r[32];
    tmem_ld32((which ? tdK : tdV) + lanebase + cc, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = key < T ? __uint_as_float(r[i]) : 0.f;
    if (key < T)
      store_row32_bf16(dqkv + ((int64_t)b * T + key) * C3 + (which ? C : 2 * C) + h * AT_HS + cc, v, mul);
    red[which * 256 + quarter * 64 + cc + lane] = warp_colsum32(v) * mul;
    // the block's column sums of dV and dK: one partial row of the qkv bias
    // gradient per (batch row, key block)
    named_bar_sync(1, DKV_CWARPS * 32);
    if (tid < 128) {
      const int wh = tid >> 6, col = tid & 63;  // 0: dV, 1: dK
      const float* rr = red + wh * 256 + col;
      const float sum = (rr[0] + rr[64]) + (rr[128] + rr[192]);
      bias_partial[((int64_t)b * gridDim.y + kb) * C3 + (wh ? C : 2 * C) + h * AT_HS + col] = sum;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == DKV_CWARPS) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

// ============================================================ backward: dQ
// One CTA per (128-query block, b*h), keys walked in 64-row sub-blocks; two
// CTAs share an SM.  Warps 0..7 compute, warp 8 (one thread) issues every
// TMA load and MMA:
//   S(j) = q k(j)^T and dP(j) = dO v(j)^T into TMEM (one buffer: the
//          compute warps copy it to registers first thing, so S(j+1) runs
//          during the elementwise work of sub-block j);
//   dQ += dS(j) k(j) once dS(j) is in shared memory (two dS buffers).
// k streams through a three-stage ring (a stage is read by S(j) and by
// dQ(j)), v through a two-stage one.
// TMEM: S 0..63, dP 64..127, dQ 128..191 (256 columns).
// smem: Q | dO | K ring | V ring (64-row tiles) | dS [2] ([128 x 64]) | barriers
#define AQ_K_STAGES 3
#define AQ_V_STAGES 2
#define AQ_THREADS (AT_THREADS + 32)
#define AQ_SMEM (1024 + 2 * AT_TILE + (AQ_K_STAGES + AQ_V_STAGES) * AT_SUBTILE + 2 * AT_TILE + 256)

__global__ void __launch_bounds__(AQ_THREADS, 2)
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
  uint8_t* sK = sm + 2 * AT_TILE;              // [AQ_K_STAGES] x [64 x 64]
  uint8_t* sV = sK + AQ_K_STAGES * AT_SUBTILE; // [AQ_V_STAGES]
  uint8_t* sS = sV + AQ_V_STAGES * AT_SUBTILE; // dS [2] x [128 queries x 64 keys]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + 2 * AT_TILE);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                 // [AQ_K_STAGES]
  uint64_t* k_empty = k_full + AQ_K_STAGES;    // [AQ_K_STAGES]: dQ(j) has read k(j)
  uint64_t* v_full = k_empty + AQ_K_STAGES;    // [AQ_V_STAGES]
  uint64_t* s_full = v_full + AQ_V_STAGES;     // S(j), dP(j) in TMEM
  uint64_t* s_empty = s_full + 1;              // 8 warps have copied them out
  uint64_t* p_full = s_empty + 1;              // [2]: 8 warps have written dS(j)
  uint64_t* p_empty = p_full + 2;              // [2]: dQ(j) has read dS(j)
  uint64_t* dq_done = p_empty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(dq_done + 1);

  const int nqb = gridDim.y;
  const int qb = nqb - 1 - blockIdx.y;  // the grid starts with the blocks that meet the most keys
  const int bh = blockIdx.x, b = bh / NH, h = bh % NH;
  const int q0 = qb * AT_BLK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsub = (min(q0 + AT_BLK, T) + AB_SUB - 1) / AB_SUB;  // key sub-blocks up to the last query

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < AQ_K_STAGES; s++) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < AQ_V_STAGES; s++) mbar_init(&v_full[s], 1);
    mbar_init(s_full, 1);
    mbar_init(s_empty, AT_THREADS / 32);
    for (int i = 0; i < 2; i++) { mbar_init(&p_full[i], AT_THREADS / 32); mbar_init(&p_empty[i], 1); }
    mbar_init(dq_done, 1);
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA + MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
      const uint32_t idO = tc_idesc_bf16(128, 64, false, true);
      auto load_k = [&](int j) {
        const int s = j % AQ_K_STAGES;
        mbar_arrive_expect_tx(&k_full[s], AT_SUBTILE);
        tma_load_3d(sK + s * AT_SUBTILE, &tm_qkv64, &k_full[s], C + h * AT_HS, j * AB_SUB, b);
      };
      auto load_v = [&](int j) {
        const int s = j % AQ_V_STAGES;
        mbar_arrive_expect_tx(&v_full[s], AT_SUBTILE);
        tma_load_3d(sV + s * AT_SUBTILE, &tm_qkv64, &v_full[s], 2 * C + h * AT_HS, j * AB_SUB, b);
      };
      auto issue_sdp = [&](int j) {  // S(j), dP(j)
        const int ks = j % AQ_K_STAGES, vs = j % AQ_V_STAGES;
        mbar_wait(&k_full[ks], (uint32_t)(j / AQ_K_STAGES) & 1u, err);
        mbar_wait(&v_full[vs], (uint32_t)(j / AQ_V_STAGES) & 1u, err);
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ), aD = smem_u32(sD);
        const uint32_t bK = smem_u32(sK + ks * AT_SUBTILE), bV = smem_u32(sV + vs * AT_SUBTILE);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tS, kmaj(aQ, kk), kmaj(bK, kk), idS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdP, kmaj(aD, kk), kmaj(bV, kk), idS, kk > 0);
        tc_commit(s_full);
      };
      mbar_arrive_expect_tx(q_full, 2 * AT_TILE);
      tma_load_3d(sQ, &tm_qkv, q_full, h * AT_HS, q0, b);
      tma_load_3d(sD, &tm_dy, q_full, h * AT_HS, q0, b);
      for (int j = 0; j < AQ_K_STAGES && j < nsub; j++) load_k(j);
      for (int j = 0; j < AQ_V_STAGES && j < nsub; j++) load_v(j);
      mbar_wait(q_full, 0, err);
      issue_sdp(0);
      for (int j = 0; j < nsub; j++) {
        if (j + 1 < nsub) {
          mbar_wait(s_empty, (uint32_t)j & 1u, err);  // S(j), dP(j) copied out (so dP(j) is done)
          if (j + AQ_V_STAGES < nsub) load_v(j + AQ_V_STAGES);
          issue_sdp(j + 1);
        }
        mbar_wait(&p_full[j & 1], (uint32_t)(j >> 1) & 1u, err);  // dS(j) written
        tc_fence_after();
        {
          const int ks = j % AQ_K_STAGES;
          const uint32_t aS = smem_u32(sS + (j & 1) * AT_TILE), bK = smem_u32(sK + ks * AT_SUBTILE);
#pragma unroll
          for (int kk = 0; kk < 4; kk++) tc_mma_bf16(tdQ, kmaj(aS, kk), mnmaj(bK, kk), idO, (j > 0 || kk > 0));
          tc_commit(&p_empty[j & 1]);
          tc_commit(&k_empty[ks]);
        }
        if (j >= 1 && j + 2 < nsub) {  // dQ(j-1) has read k(j-1): its stage takes k(j+2)
          mbar_wait(&k_empty[(j - 1) % AQ_K_STAGES], (uint32_t)((j - 1) / AQ_K_STAGES) & 1u, err);
          load_k(j + 2);
        }
      }
      tc_commit(dq_done);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane, q = q0 + row;
    const uint32_t lanebase = (uint32_t)(quarter * 32) << 16;
    const float sl2 = scale * 1.4426950408889634f;
    const float my_lse = q < T ? lse[(int64_t)bh * T + q] : INFINITY;  // base 2
    const float my_d = q < T ? dsum[(int64_t)bh * T + q] : 0.f;
    for (int j = 0; j < nsub; j++) {
      const int k0 = j * AB_SUB;
      mbar_wait(s_full, (uint32_t)j & 1u, err);
      tc_fence_after();
      uint32_t rs[32], rd[32];
      tmem_ld32(tS + lanebase + half * 32, rs);
      tmem_ld32(tdP + lanebase + half * 32, rd);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      mbar_wait(&p_empty[j & 1], ((uint32_t)(j >> 1) & 1u) ^ 1u, err);  // dQ(j-2) has read the buffer
      uint8_t* srow = sS + (j & 1) * AT_TILE + row * 128;
      if (k0 + AB_SUB > q0)
        qrow_elementwise<true>(rs, rd, my_lse, my_d, sl2, k0 + half * 32, q, srow, row & 7, half * 4);
      else
        qrow_elementwise<false>(rs, rd, my_lse, my_d, sl2, k0 + half * 32, q, srow, row & 7, half * 4);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
    }
    mbar_wait(dq_done, 0, err);
    tc_fence_after();
    float v[32];
    {
      uint32_t r[32];
      tmem_ld32(tdQ + lanebase + half * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = q < T ? __uint_as_float(r[i]) : 0.f;
    }
    if (q < T) store_row32_bf16(dqkv + ((int64_t)b * T + q) * 3 * (int64_t)C + h * AT_HS + half * 32, v, scale);
    // the block's column sums of dQ: one partial row of the qkv bias gradient
    // per (batch row, query block); the dS buffers are free once dQ is done
    float* red = reinterpret_cast<float*>(sS);  // [4][64]
    red[quarter * 64 + half * 32 + lane] = warp_colsum32(v) * scale;
    named_bar_sync(1, AT_THREADS);
    if (tid < 64) {
      const float* rr = red + tid;
      bias_partial[((int64_t)b * nqb + qb) * 3 * (int64_t)C + h * AT_HS + tid] = (rr[0] + rr[64]) + (rr[128] + rr[192]);
    }
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
  CUtensorMap tq, td, tq64;
  if (!make_tmap_btw(&tq, qkv, B, T, 3 * C) || !make_tmap_btw(&td, dy, B, T, C) ||
      !make_tmap_btw(&tq64, qkv, B, T, 3 * C, AB_SUB)) {
    c.host_fail = 1;
    return false;
  }
  const int64_t n = (int64_t)B * T * NH;
  launch_pdl(c, attn_bwd_dsum_kernel, dim3((int)std::min<int64_t>((n + 255) / 256, (int64_t)c.num_sms * 16)), dim3(256), 0, dsum, dy, y, B, T, C, NH);
  const float scale = 1.f / sqrtf((float)AT_HS);
  dim3 grid(B * NH, (T + AT_BLK - 1) / AT_BLK);
  const size_t kv_smem = akv_smem(T);
  cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kv_smem);
  launch_pdl(c, attn_bwd_dkv_tc_kernel, dim3(grid), dim3(DKV_THREADS), kv_smem, tq, td, dqkv, lse, dsum, bias_partial, T, C, NH, scale, c.err);
  cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AQ_SMEM);
  launch_pdl(c, attn_bwd_dq_tc_kernel, dim3(grid), dim3(AQ_THREADS), AQ_SMEM, tq, td, tq64, dqkv, lse, dsum, bias_partial, T, C, NH, scale, c.err);
  return true;
}
