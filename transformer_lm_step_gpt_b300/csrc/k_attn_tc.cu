// k_attn_tc.cu -- causal multi-head self-attention on the tcgen05 tensor cores.
//
// GeekNews, "A GPT-2-based ChatGPT clone in 3000 bytes of C", section "The
// Transformer core": per head, S = q k^T (scaled by 1/sqrt(hs)), the lower-
// triangular causal mask, softmax over each query row, times v.  Here the
// T x T score matrix is never stored: it is computed one 128 x 128 block at
// a time in tensor memory (TMEM), folded into an online softmax (forward) or
// recomputed from the saved row logsumexp (backward).
//
// Head sizes 16, 32, 64 and 128.  Every tile of q, k, v, dy is one or two
// TMA boxes [rows x 64 columns] of a 3-D tensor map over [B, T, width] (rows
// past T read as zero), 128-byte swizzled in shared memory, where a tcgen05
// descriptor reads it either as a K-major operand (rows = M or N, K = head
// dims) or as an MN-major one (rows = K).  Head sizes below 64 load the
// full 64-column box (the extra columns are never multiplied).  The
// probabilities P and the score gradients dS never go to shared memory:
// the elementwise warps write them into TMEM as packed bf16 pairs, where
// the next product reads them as its A operand.
//
// The tensor pipe takes about 71 cycles for one M = 128, K = 16 product at
// N = 64 and at N = 128, and 128 cycles at N = 256 (measured on this B300),
// so every score product here has N = 128 keys (or queries): 128-key blocks.
//
// All three kernels are persistent: a CTA walks a fixed list of work items
// (a query block or key block of one (batch, head)), longest first and
// assigned in a snake order over the grid, and the roles run ahead across
// item boundaries (the next item's loads and score products start while
// this item's last elementwise step and epilogue run).  Roles per CTA: one
// TMA loader thread, one MMA issuer thread, 8 or 16 elementwise warps; every
// hand-off is an mbarrier; every wait is bounded (common.cuh) and a wait that
// gives up records a timeout and the kernel runs on to its end.
//
//   forward  item (128-query block, b*h), 128-key blocks: S(j) = q k(j)^T in
//            TMEM; the softmax warps copy it to registers (so S(j+1) runs
//            during their work), take P relative to a row reference maximum
//            that moves only when the row maximum grows by more than 2^8
//            (then O is rescaled in TMEM), write P into TMEM; O += P v(j)
//            accumulates in TMEM.  Saves minus the row logsumexp in base 2
//            (the backward adds it in one fused multiply-add).
//   dK, dV   item (128-key block, b*h), query sub-blocks of 128 (64 for head
//            size 128): S^T = k q^T and dP^T = v dy^T; P^T and dS^T =
//            P^T (dP^T - D) into TMEM; dV += P^T dy, dK += dS^T q.  D is
//            stored negated (added, not subtracted).
//   dQ       item (128-query block, b*h), 128-key blocks: S = q k^T, dP =
//            dy v^T; dS into TMEM; dQ += dS k.
// No atomics: every output element is written by one CTA, so the results
// repeat bit for bit.  At head size 64 the output tiles leave through
// shared memory, where the epilogues also take their column sums (the qkv
// bias gradient's partial rows); other head sizes leave the bias gradient
// to a column-sum pass over dqkv.
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
bool attn_tmap_btw(CUtensorMap* m, const void* base, int B, int T, int W, int rows) {
  return make_tmap_btw(m, base, B, T, W, rows);
}

#define LOG2E_F 1.4426950408889634f

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

// Tiles: R rows x HS head dims, stored as NB = ceil(HS/64) boxes of
// [R rows x 64 columns] (128 bytes per row, 128-byte swizzle), box i at
// tile + i * R * 128.
template <int HS>
struct Hs {
  static_assert(HS == 16 || HS == 32 || HS == 64 || HS == 128, "head size");
  static constexpr int NB = HS > 64 ? 2 : 1;
  static constexpr int KS = HS / 16;  // K steps of 16 over the head dims
};
// K-major operand (rows = M or N, K = head dims), K step kk
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int rows, int kk) {
  return sw128_desc(tile + (uint32_t)((kk >> 2) * rows * 128 + (kk & 3) * 32), 16, 1024);
}
// MN-major operand (rows = K, head dims = N), K step kk (16 rows); the
// 64-column boxes are rows*128 bytes apart
__device__ __forceinline__ uint64_t ndesc(uint32_t tile, int rows, int kk) {
  return sw128_desc(tile + (uint32_t)(kk * 2048), (uint32_t)(rows * 128), 1024);
}
// The same descriptors as a base (K step 0) plus a constant: the start
// address field holds address / 16 in the low bits, so a K step adds its
// byte offset / 16 to the 64-bit descriptor
__device__ __forceinline__ uint64_t kstep(int rows, int kk) {
  return (uint64_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t nstep(int kk) { return (uint64_t)(kk * 128); }
// A chain of K steps over the head dims (KS = HS/16) of two K-major
// shared-memory operands with `arows` and `brows` rows: four steps per
// statement while at least four remain in a 64-column box.
template <int KS>
__device__ __forceinline__ void mma_hs_ss(uint32_t d, uint64_t a, int arows, uint64_t b, int brows, uint32_t idesc) {
  if constexpr (KS >= 4) {
#pragma unroll
    for (int c = 0; c < KS / 4; c++)
      tc_mma4_ss<2, 2>(d, a + kstep(arows, 4 * c), b + kstep(brows, 4 * c), idesc, c > 0 ? 1u : 0u);
  } else {
#pragma unroll
    for (int kk = 0; kk < KS; kk++) tc_mma_bf16(d, a + kstep(arows, kk), b + kstep(brows, kk), idesc, kk > 0 ? 1u : 0u);
  }
}
// A chain of NK K steps (a multiple of 4, or 1 or 2) with A in TMEM from
// column a (8 columns of bf16 pairs per step) and an MN-major B operand
// (K = rows): dst (+)= A B, accumulating iff acc.
template <int NK>
__device__ __forceinline__ void mma_ts_chain(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, bool acc) {
  if constexpr (NK % 4 == 0) {
#pragma unroll
    for (int c = 0; c < NK / 4; c++) tc_mma4_ts<128>(d, a + 32 * c, b + nstep(4 * c), idesc, (acc || c > 0) ? 1u : 0u);
  } else {
    static_assert(NK == 1 || NK == 2, "K steps");
#pragma unroll
    for (int kk = 0; kk < NK; kk++) tc_mma_bf16_ts(d, a + 8 * kk, b + nstep(kk), idesc, (acc || kk > 0) ? 1u : 0u);
  }
}
// TMA of one tile (NB boxes) onto one barrier
template <int HS>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col,
                                          int row, int b, int rows) {
#pragma unroll
  for (int i = 0; i < Hs<HS>::NB; i++) tma_load_3d(dst + i * rows * 128, map, bar, col + 64 * i, row, b);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}
// N floats (N a multiple of 8) times mul as bf16 to 16-byte aligned global memory
template <int N>
__device__ __forceinline__ void store_bf16_row(bf16* dst, const float* v, float mul) {
#pragma unroll
  for (int i = 0; i < N; i += 8) {
    uint4 u;
    u.x = pack_bf16(v[i] * mul, v[i + 1] * mul);
    u.y = pack_bf16(v[i + 2] * mul, v[i + 3] * mul);
    u.z = pack_bf16(v[i + 4] * mul, v[i + 5] * mul);
    u.w = pack_bf16(v[i + 6] * mul, v[i + 7] * mul);
    *reinterpret_cast<uint4*>(dst + i) = u;
  }
}
// Sum over the 32 lanes of each of N values; every lane gets the sums.
template <int N>
__device__ __forceinline__ void warp_sum_cols(float* v) {
#pragma unroll
  for (int i = 0; i < N; i++) v[i] = warp_sum(v[i]);
}

// The persistent schedule: round r of CTA c takes item r*G + c (r even) or
// r*G + G-1-c (r odd), so the longest items (first in the list) spread over
// the grid and each CTA's total stays close to the mean.
__device__ __forceinline__ int snake_item(int r) {
  const int G = gridDim.x, c = blockIdx.x;
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// ============================================================ forward
// Warps 0..7 softmax (warps w and w+4 share TMEM lane quarter w % 4, i.e. 32
// query rows, and take key columns 0..63 / 64..127 of a block and head dims
// 0..HS/2-1 / HS/2..HS-1 of O), warp 8 the MMA issuer, warp 9 the loader.
// TMEM: S 0..127, P 128..191 (bf16 pairs), O 192..192+HS-1.
// smem: Q [QB] | K ring [2] | V ring [2] | y staging (head size 64) |
//       row-max exchange [2][2][128] | row-sum exchange [2][128] | barriers.
#define FW_SOFT 8
#define FW_THREADS (FW_SOFT * 32 + 64)
template <int HS>
struct FwdCfg {
  static constexpr uint32_t TILE = Hs<HS>::NB * 16384u;  // [128 x HS]
  // head size 64: the y tile leaves through a shared-memory staging tile and
  // one TMA store; to fit it next to a second CTA on the SM, one q buffer
  static constexpr bool STAGE_OUT = HS == 64;
  static constexpr int QB = STAGE_OUT ? 1 : 2, KV = 2;
  static constexpr int TMEM = HS > 64 ? 512 : 256;
  static constexpr int PER_SM = HS > 64 ? 1 : 2;
  static constexpr uint32_t OUT_BYTES = STAGE_OUT ? 16384u : 0u;
  static constexpr uint32_t SMEM = 1024 + (QB + 2 * KV) * TILE + OUT_BYTES + 2048 + 1024 + 256;
};

template <int HS>
__global__ void __launch_bounds__(FW_THREADS, FwdCfg<HS>::PER_SM)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_y,
                       bf16* y, float* lse, int B, int T, int C, int NH, float scale, int* err) {
  using Cf = FwdCfg<HS>;
  constexpr int QB = Cf::QB, KV = Cf::KV;
  constexpr uint32_t TILE = Cf::TILE;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + QB * TILE;
  uint8_t* sV = sK + KV * TILE;
  uint8_t* sOut = sV + KV * TILE;                          // y staging (head size 64)
  float* red = reinterpret_cast<float*>(sOut + Cf::OUT_BYTES);  // [2][2][128]
  float* lred = red + 512;                                 // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(lred + 256);
  uint64_t* q_full = bars;             // [QB]
  uint64_t* q_empty = q_full + QB;     // [QB]: the item's last S has read Q
  uint64_t* k_full = q_empty + QB;     // [KV]
  uint64_t* k_empty = k_full + KV;     // [KV]
  uint64_t* v_full = k_empty + KV;     // [KV]
  uint64_t* v_empty = v_full + KV;     // [KV]
  uint64_t* s_full = v_empty + KV;     // S(g) in TMEM
  uint64_t* s_free = s_full + 1;       // the softmax warps have copied S(g) out
  uint64_t* p_full = s_free + 1;       // the softmax warps have written P(g)
  uint64_t* o_done = p_full + 1;       // P(g) V(g) complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(o_done + 1);

  const int nqb = (T + 127) / 128, BH = B * NH, nitems = nqb * BH;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < QB; i++) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < KV; i++) {
      mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, FW_SOFT);
    mbar_init(p_full, FW_SOFT);
    mbar_init(o_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
  }
  if (warp == 0) { tmem_alloc(tslot, Cf::TMEM); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_trigger();  // dependents launch only once every CTA holds its tensor memory
  pdl_wait();     // from here on global memory written by the previous kernel is read
  const uint32_t tS = tm, tP = tm + 128, tO = tm + 192;

  if (warp == FW_SOFT) {
    // ------------------------------------------------------------ MMA issuer
    // (one thread: a second issuer warp would cost the softmax warps the
    // registers that two CTAs per SM leave them)
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 128, false, false);
      const uint32_t idO = tc_idesc_bf16(128, HS, false, true);
      auto pv = [&](int gp, bool first) {  // O (+)= P(gp) v(gp), P from TMEM
        mbar_wait(p_full, (uint32_t)gp & 1u, err);
        mbar_wait(&v_full[gp % KV], (uint32_t)(gp / KV) & 1u, err);
        tc_fence_after();
        const uint64_t dV = ndesc(smem_u32(sV + (gp % KV) * TILE), 128, 0);
        mma_ts_chain<8>(tO, tP, dV, idO, !first);
        tc_commit(&v_empty[gp % KV]);
        tc_commit(o_done);
      };
      int g = 0, it = 0;
      bool prev = false, prev_first = false;
      for (int r = 0;; r++, it++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int nk = nqb - idx / BH;  // key blocks 0 .. qb
        const int qs = it % QB;
        mbar_wait(&q_full[qs], (uint32_t)(it / QB) & 1u, err);
        const uint64_t dQ = kdesc(smem_u32(sQ + qs * TILE), 128, 0);
        for (int j = 0; j < nk; j++, g++) {
          mbar_wait(&k_full[g % KV], (uint32_t)(g / KV) & 1u, err);
          if (g > 0) mbar_wait(s_free, (uint32_t)(g - 1) & 1u, err);
          tc_fence_after();
          const uint64_t dK = kdesc(smem_u32(sK + (g % KV) * TILE), 128, 0);
          mma_hs_ss<Hs<HS>::KS>(tS, dQ, 128, dK, 128, idS);
          tc_commit(&k_empty[g % KV]);
          if (j == nk - 1) tc_commit(&q_empty[qs]);
          tc_commit(s_full);
          if (prev) pv(g - 1, prev_first);  // the previous block's PV runs after this S
          prev = true;
          prev_first = j == 0;
        }
      }
      if (prev) pv(g - 1, prev_first);
    }
  } else if (warp == FW_SOFT + 1) {
    // ------------------------------------------------------------ TMA loader
    if (lane == 0) {
      int g = 0, it = 0;
      for (int r = 0;; r++, it++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int qb = nqb - 1 - idx / BH, bh = idx % BH, b = bh / NH, h = bh % NH;
        const int qs = it % QB;
        if (it >= QB) mbar_wait(&q_empty[qs], (uint32_t)(it / QB - 1) & 1u, err);
        mbar_arrive_expect_tx(&q_full[qs], TILE);
        load_tile<HS>(sQ + qs * TILE, &tm_qkv, &q_full[qs], h * HS, qb * 128, b, 128);
        for (int j = 0; j <= qb; j++, g++) {
          const int s = g % KV;
          if (g >= KV) mbar_wait(&k_empty[s], (uint32_t)(g / KV - 1) & 1u, err);
          mbar_arrive_expect_tx(&k_full[s], TILE);
          load_tile<HS>(sK + s * TILE, &tm_qkv, &k_full[s], C + h * HS, j * 128, b, 128);
          if (g >= KV) mbar_wait(&v_empty[s], (uint32_t)(g / KV - 1) & 1u, err);
          mbar_arrive_expect_tx(&v_full[s], TILE);
          load_tile<HS>(sV + s * TILE, &tm_qkv, &v_full[s], 2 * C + h * HS, j * 128, b, 128);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const float sl2 = scale * LOG2E_F;  // scores -> log2 units
    constexpr int OH = HS / 2;          // O columns of this warp
    int g = 0;
    for (int r = 0;; r++) {
      const int idx = snake_item(r);
      if (idx >= nitems) break;
      const int qb = nqb - 1 - idx / BH, bh = idx % BH, b = bh / NH, h = bh % NH;
      const int q = qb * 128 + row, nk = qb + 1;
      // m: the row's reference maximum (raw score units); P and the row sum
      // are relative to it; it moves only when a block's maximum exceeds it
      // by more than 8 in log2 units, and then O and the sum are rescaled
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nk; j++, g++) {
        mbar_wait(s_full, (uint32_t)g & 1u, err);
        tc_fence_after();
        uint32_t s[64];
        tmem_ld32(tS + lb + half * 64, *reinterpret_cast<uint32_t(*)[32]>(s));
        tmem_ld32(tS + lb + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        const int k0 = j * 128 + half * 64;  // key of column 0 of this warp
        if (j == nk - 1) {  // the diagonal block: keys after the query read as -inf
#pragma unroll
          for (int c = 0; c < 64; c++)
            if (k0 + c > q) s[c] = __float_as_uint(-INFINITY);
        }
        float mx;
        {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 64; c += 8)
#pragma unroll
            for (int u = 0; u < 4; u++)
              m4[u] = fmax3(m4[u], __uint_as_float(s[c + 2 * u]), __uint_as_float(s[c + 2 * u + 1]));
          mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        }
        float* rd = red + (g & 1) * 256;
        rd[half * 128 + row] = mx;
        named_bar_sync(1 + quarter, 64);  // warps quarter and quarter + 4
        const float mcand = fmaxf(m, fmaxf(rd[row], rd[128 + row]));
        const bool resc = (mcand - m) * sl2 > 8.f;  // always at j = 0 (m = -inf)
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_hw((m - mcand) * sl2);
          l *= alpha;
          m = mcand;
        }
        // p = 2^(s sl2 - m sl2), two columns per instruction
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nmo2 = f2_pack(-m * sl2, -m * sl2);
        uint64_t sum2 = f2_pack(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, nmo2), x0, x1);
          const float p0 = ex2_hw(x0), p1 = ex2_hw(x1);
          sum2 = f2_add(sum2, f2_pack(p0, p1));
          pk[c >> 1] = pack_bf16(p0, p1);
        }
        float sa, sb;
        f2_unpack(sum2, sa, sb);
        const float sum = sa + sb;
        if (j > 0) {
          // P(g-1) V(g-1) done: the P columns are free and O is complete up
          // to block g-1 (at j = 0 the previous item's epilogue waited)
          mbar_wait(o_done, (uint32_t)(g - 1) & 1u, err);
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
            uint32_t o[OH];
            tmem_ld_cols<OH>(tO + lb + half * OH, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < OH; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_cols<OH>(tO + lb + half * OH, o);
          }
        }
        l += sum;
        tmem_st16(tP + lb + half * 32, pk);
        tmem_st16(tP + lb + half * 32 + 16, pk + 16);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      // epilogue: O = sum over blocks of P V, relative to the final maximum
      mbar_wait(o_done, (uint32_t)(g - 1) & 1u, err);
      tc_fence_after();
      uint32_t o[OH];
      tmem_ld_cols<OH>(tO + lb + half * OH, o);
      tmem_ld_wait();
      lred[half * 128 + row] = l;
      named_bar_sync(1 + quarter, 64);
      const float lt = lred[row] + lred[128 + row];
      if (q < T && half == 0) lse[(int64_t)bh * T + q] = -(m * sl2 + log2f(lt));  // minus lse, base-2 units
      if constexpr (Cf::STAGE_OUT) {
        // the warp's 32 rows x 32 columns into the 128B-swizzled staging
        // tile (16-byte chunks 4 half .. 4 half + 3 of each row), then one
        // TMA store of the [128 x 64] tile (rows past T are not written);
        // the previous item's store has read the tile before it is rewritten
        if (tid == 0) bulk_wait_read0();
        named_bar_sync(5, FW_SOFT * 32);
        const float inv = 1.f / lt;
        uint8_t* rowp = sOut + row * 128;
#pragma unroll
        for (int qq = 0; qq < 4; qq++) {
          uint4 u;
          u.x = pack_bf16(__uint_as_float(o[8 * qq]) * inv, __uint_as_float(o[8 * qq + 1]) * inv);
          u.y = pack_bf16(__uint_as_float(o[8 * qq + 2]) * inv, __uint_as_float(o[8 * qq + 3]) * inv);
          u.z = pack_bf16(__uint_as_float(o[8 * qq + 4]) * inv, __uint_as_float(o[8 * qq + 5]) * inv);
          u.w = pack_bf16(__uint_as_float(o[8 * qq + 6]) * inv, __uint_as_float(o[8 * qq + 7]) * inv);
          *reinterpret_cast<uint4*>(rowp + (((half * 4 + qq) ^ (row & 7)) << 4)) = u;
        }
        fence_proxy_async_smem();
        named_bar_sync(5, FW_SOFT * 32);
        if (tid == 0) {
          tma_store_3d(&tm_y, sOut, h * HS, qb * 128, b);
          bulk_commit();
        }
      } else if (q < T) {
        float v[OH];
#pragma unroll
        for (int i = 0; i < OH; i++) v[i] = __uint_as_float(o[i]);
        store_bf16_row<OH>(y + ((int64_t)b * T + q) * C + h * HS + half * OH, v, 1.f / lt);
      }
    }
  }
  if (Cf::STAGE_OUT && tid == 0) bulk_wait0();  // the last item's store is complete
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tm, Cf::TMEM); }
}

// ============================================================ backward: D
// D[b,h,t] = sum_i dy[b,t,h*HS+i] * y[b,t,h*HS+i].  Thread i takes the
// 16-byte chunk i of the [B*T, C] rows (coalesced), the HS/8 threads of one
// head add their partial dots with shuffles, the first writes D.
template <int HS>
__global__ void attn_bwd_dsum_kernel(float* dsum, const bf16* dy, const bf16* y, int B, int T, int C,
                                     int NH) {
  pdl_trigger();
  pdl_wait();
  constexpr int G = HS / 8;  // threads per head
  const int chunks = C / 8;
  const int64_t n = (int64_t)B * T * chunks;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x; i0 < n; i0 += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = i0 + threadIdx.x;
    float s = 0.f;
    if (i < n) {
      const uint4 ua = reinterpret_cast<const uint4*>(dy)[i];
      const uint4 uc = reinterpret_cast<const uint4*>(y)[i];
      const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wc[4] = {uc.x, uc.y, uc.z, uc.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[j]));
        const float2 fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wc[j]));
        s += fa.x * fc.x + fa.y * fc.y;
      }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (i < n && (i % G) == 0) {
      const int64_t bt = i / chunks;
      const int h = (int)(i % chunks) / G;
      const int t = (int)(bt % T), b = (int)(bt / T);
      dsum[((int64_t)b * NH + h) * T + t] = -s;
    }
  }
}

// Column sums of R rows (from r0, a multiple of 8) of a 128B-swizzled
// [rows x 64] bf16 staging tile: lane l adds columns 2l and 2l + 1; rows at
// or past `valid` count 0.  Full row groups take the unrolled loop with
// constant swizzle offsets and f32x2 adds.
template <int R>
__device__ __forceinline__ float2 tile_colsum2(const uint8_t* tile, int r0, int valid, int lane) {
  const int cb = lane >> 2, co = (lane & 3) * 4;
  const uint8_t* base = tile + r0 * 128 + co;
  uint64_t s = f2_pack(0.f, 0.f);
  if (r0 + R <= valid) {
#pragma unroll 8
    for (int i = 0; i < R; i++) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(base + i * 128 + ((cb ^ (i & 7)) << 4));
      s = f2_add(s, f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)));
    }
  } else {
#pragma unroll 4
    for (int i = 0; i < R; i++) {
      if (r0 + i < valid) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(base + i * 128 + ((cb ^ (i & 7)) << 4));
        s = f2_add(s, f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)));
      }
    }
  }
  float2 o;
  f2_unpack(s, o.x, o.y);
  return o;
}

// ============================================================ backward: dK, dV
// The elementwise step of one key row over N query columns (c0 .. c0+N-1):
// P^T = 2^(S^T sl2 - lse2), dS^T = P^T (dP^T - D), packed to bf16 pairs.
// nl, nd: minus lse2 and minus D of the columns, from shared memory
// (STAGED) or global memory (gl, gd: the (b, h) rows, read at c0 + i).
// MASK: columns before the key or past T give 0 (a masked column may hold
// a stale lse / D: select, do not scale).  Each combination is its own
// instantiation, so that sub-blocks off the diagonal carry no
// compare-and-select and the staged path no global-load addressing.
template <int N, bool MASK, bool STAGED>
__device__ __forceinline__ void kv_elementwise(const uint32_t* rs, const uint32_t* rd, const float* nl, const float* nd,
                                               const float* gl, const float* gd, int c0, int key, int T,
                                               float sl2, uint32_t* pk, uint32_t* dk) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    float4 a, d;
    if (STAGED) {
      a = *reinterpret_cast<const float4*>(nl + i);
      d = *reinterpret_cast<const float4*>(nd + i);
    } else {
      float t[8];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int qq = min(c0 + i + u, T - 1);
        t[u] = __ldg(gl + qq);
        t[4 + u] = __ldg(gd + qq);
      }
      a = make_float4(t[0], t[1], t[2], t[3]);
      d = make_float4(t[4], t[5], t[6], t[7]);
    }
    float x0, x1, x2, x3;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[i]), __uint_as_float(rs[i + 1])), sl2x2, f2_pack(a.x, a.y)), x0, x1);
    f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[i + 2]), __uint_as_float(rs[i + 3])), sl2x2, f2_pack(a.z, a.w)), x2, x3);
    float p0 = ex2_hw(x0), p1 = ex2_hw(x1), p2 = ex2_hw(x2), p3 = ex2_hw(x3);
    const uint64_t t01 = f2_add(f2_pack(__uint_as_float(rd[i]), __uint_as_float(rd[i + 1])), f2_pack(d.x, d.y));
    const uint64_t t23 = f2_add(f2_pack(__uint_as_float(rd[i + 2]), __uint_as_float(rd[i + 3])), f2_pack(d.z, d.w));
    float d0, d1, d2, d3;
    f2_unpack(f2_mul(f2_pack(p0, p1), t01), d0, d1);
    f2_unpack(f2_mul(f2_pack(p2, p3), t23), d2, d3);
    if (MASK) {
      const int c = c0 + i;
      const bool ok0 = c >= key && c < T, ok1 = c + 1 >= key && c + 1 < T;
      const bool ok2 = c + 2 >= key && c + 2 < T, ok3 = c + 3 >= key && c + 3 < T;
      p0 = ok0 ? p0 : 0.f; d0 = ok0 ? d0 : 0.f;
      p1 = ok1 ? p1 : 0.f; d1 = ok1 ? d1 : 0.f;
      p2 = ok2 ? p2 : 0.f; d2 = ok2 ? d2 : 0.f;
      p3 = ok3 ? p3 : 0.f; d3 = ok3 ? d3 : 0.f;
    }
    pk[i >> 1] = pack_bf16(p0, p1);
    pk[(i >> 1) + 1] = pack_bf16(p2, p3);
    dk[i >> 1] = pack_bf16(d0, d1);
    dk[(i >> 1) + 1] = pack_bf16(d2, d3);
  }
}

// Item (128-key block kb, b*h): query sub-blocks of QS rows from k0 = 128 kb
// to T, each taken in two column halves of QS/2 queries.  Warps 0..15
// elementwise in two groups: group h (warps 8h..8h+7) owns half h of every
// sub-block (warps w and w+4 of a group share TMEM lane quarter w % 4 = 32
// key rows and take QS/4 query columns each); warp 16 issues the score
// products, warp 17 loads, warp 18 issues the gradient products.
//   S^T = k q^T, dP^T = v dy^T (M = 128 keys, N = QS/2 queries per half, K = HS);
//   P^T = 2^(S^T scale log2e - lse2), dS^T = P^T (dP^T - D), into TMEM;
//   dV += P^T dy, dK += dS^T q (N = HS, K = QS/2 queries per half; A from TMEM).
// Each half has its own hand-offs (scores in, scores copied out, P^T / dS^T
// in, P^T / dS^T read), so one group's TMEM loads and arithmetic overlap the
// other group's, and the tensor pipe works on one half while the warps
// work on the other.  The item's epilogue is group 0's, one item late.
// TMEM: S^T 0..QS-1, dP^T QS..2QS-1, P^T 2QS.., dS^T 2.5QS.., dV 3QS..,
// dK 3QS+HS.. (at most 512 columns).
// smem: K, V [KVB] | q, dy ring [ST] | lse / D per stage [ST][2][QS] | barriers.
// lse and D of a sub-block arrive by bulk copy with its tiles when T is a
// multiple of 4 (16-byte aligned rows); otherwise the elementwise warps read
// them from global memory.
#define KV_CW 16
#define KV_GW 8  // warps per elementwise group
#define KV_THREADS (KV_CW * 32 + 96)
template <int HS>
struct KvCfg {
  static constexpr int QS = HS > 64 ? 64 : 128;
  static constexpr int QH = QS / 2;   // queries per half
  static constexpr int CPT = QS / 4;  // query columns per elementwise thread
  static constexpr uint32_t KTILE = Hs<HS>::NB * 16384u;                  // [128 x HS]
  static constexpr uint32_t QTILE = Hs<HS>::NB * (uint32_t)QS * 128u;     // [QS x HS]
  static constexpr int KVB = HS > 64 ? 1 : 2;
  // head size 64: dV and dK tiles ([128 x 64] bf16 each) leave through a
  // shared-memory staging area and one TMA store each (three ring stages
  // leave room for it); other head sizes store rows directly
  static constexpr bool STAGE_OUT = HS == 64;
  static constexpr int ST = STAGE_OUT ? 3 : 4;
  static constexpr uint32_t OUT_BYTES = STAGE_OUT ? 2 * 16384u : 0u;
  static constexpr uint32_t RED_BYTES = STAGE_OUT ? 2 * 4 * 64 * 4 : 0u;  // column-sum partials [2][4][64]
  static constexpr uint32_t SMEM = 1024 + KVB * 2 * KTILE + ST * 2 * QTILE + ST * 2 * QS * 4 + OUT_BYTES + RED_BYTES + 256;
};

template <int HS, bool STAGED>
__global__ void __launch_bounds__(KV_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                           const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_out,
                           bf16* dqkv, const float* lse, const float* dsum, float* bias_partial, int B, int T, int C,
                           int NH, float scale, int* err) {
  using Cf = KvCfg<HS>;
  constexpr int QS = Cf::QS, QH = Cf::QH, CPT = Cf::CPT, KVB = Cf::KVB, ST = Cf::ST;
  constexpr uint32_t KTILE = Cf::KTILE, QTILE = Cf::QTILE;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sK = sm;                          // [KVB]
  uint8_t* sV = sK + KVB * KTILE;            // [KVB]
  uint8_t* sQ = sV + KVB * KTILE;            // [ST]
  uint8_t* sD = sQ + ST * QTILE;             // dy [ST]
  float* sLD = reinterpret_cast<float*>(sD + ST * QTILE);  // [ST][lse QS, D QS]
  uint8_t* sOut = reinterpret_cast<uint8_t*>(sLD + ST * 2 * QS);  // dV | dK staging (head size 64)
  float* red = reinterpret_cast<float*>(sOut + Cf::OUT_BYTES);     // [2][4][64] column-sum partials
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + Cf::RED_BYTES);
  uint64_t* kv_full = bars;              // [KVB]
  uint64_t* kv_empty = kv_full + KVB;    // [KVB]: the item's last S^T, dP^T have read k, v
  uint64_t* q_full = kv_empty + KVB;     // [ST]
  uint64_t* q_empty = q_full + ST;       // [ST]: dV, dK of the sub-block done
  uint64_t* s_full = q_empty + ST;       // [2] S^T, dP^T of a half in TMEM
  uint64_t* s_free = s_full + 2;         // [2] copied out by the half's group
  uint64_t* p_full = s_free + 2;         // [2] P^T, dS^T of a half written by its group
  uint64_t* p_empty = p_full + 2;        // [2] dV, dK have read them
  uint64_t* acc_full = p_empty + 2;      // the item's dV, dK complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int nkb = (T + 127) / 128, BH = B * NH, nitems = nkb * BH;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr bool staged = STAGED;  // lse, D rows 16-byte aligned: T % 4 == 0
  if (tid == 0) {
    for (int i = 0; i < KVB; i++) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 1); }
    for (int i = 0; i < ST; i++) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < 2; i++) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], KV_GW);
      mbar_init(&p_full[i], KV_GW);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_dy);
  }
  if (warp == KV_CW) { tmem_alloc(tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_trigger();  // dependents launch only once every CTA holds its tensor memory
  pdl_wait();
  const uint32_t tSt = tm, tdPt = tm + QS, tPt = tm + 2 * QS, tdSt = tm + 2 * QS + QS / 2;
  const uint32_t tdV = tm + 3 * QS, tdK = tm + 3 * QS + HS;
  const float sl2 = scale * LOG2E_F;

  if (warp == KV_CW + 1) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      int g = 0, it = 0;
      for (int r = 0;; r++, it++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int kb = idx / BH, bh = idx % BH, b = bh / NH, h = bh % NH, k0 = kb * 128;
        const int kvb = it % KVB;
        if (it >= KVB) mbar_wait(&kv_empty[kvb], (uint32_t)(it / KVB - 1) & 1u, err);
        mbar_arrive_expect_tx(&kv_full[kvb], 2 * KTILE);
        load_tile<HS>(sK + kvb * KTILE, &tm_kv, &kv_full[kvb], C + h * HS, k0, b, 128);
        load_tile<HS>(sV + kvb * KTILE, &tm_kv, &kv_full[kvb], 2 * C + h * HS, k0, b, 128);
        const int nsub = (T - k0 + QS - 1) / QS;
        for (int j = 0; j < nsub; j++, g++) {
          const int s = g % ST, q0 = k0 + j * QS;
          if (g >= ST) mbar_wait(&q_empty[s], (uint32_t)(g / ST - 1) & 1u, err);
          const uint32_t ldb = staged ? 4u * (uint32_t)min(QS, T - q0) : 0u;  // a multiple of 16
          mbar_arrive_expect_tx(&q_full[s], 2 * QTILE + 2 * ldb);
          load_tile<HS>(sQ + s * QTILE, &tm_q, &q_full[s], h * HS, q0, b, QS);
          load_tile<HS>(sD + s * QTILE, &tm_dy, &q_full[s], h * HS, q0, b, QS);
          if (staged) {
            bulk_load(sLD + s * 2 * QS, lse + (int64_t)bh * T + q0, ldb, &q_full[s]);
            bulk_load(sLD + s * 2 * QS + QS, dsum + (int64_t)bh * T + q0, ldb, &q_full[s]);
          }
        }
      }
    }
  } else if (warp == KV_CW) {
    // ---------------------------------------------------------------- score MMAs
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, QH, false, false);
      int g = 0, it = 0;
      for (int r = 0;; r++, it++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int k0 = (idx / BH) * 128;
        const int nsub = (T - k0 + QS - 1) / QS;
        const int kvb = it % KVB;
        mbar_wait(&kv_full[kvb], (uint32_t)(it / KVB) & 1u, err);
        const uint64_t dK = kdesc(smem_u32(sK + kvb * KTILE), 128, 0), dV = kdesc(smem_u32(sV + kvb * KTILE), 128, 0);
        for (int j = 0; j < nsub; j++, g++) {
          const int s = g % ST;
          mbar_wait(&q_full[s], (uint32_t)(g / ST) & 1u, err);
          const uint64_t dQ = kdesc(smem_u32(sQ + s * QTILE), QS, 0), dD = kdesc(smem_u32(sD + s * QTILE), QS, 0);
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            // half hf: query rows hf*QH.. of the stage (their 128-byte rows
            // start hf*QH*128 bytes in, a multiple of the 1 KB swizzle atom)
            if (g > 0) mbar_wait(&s_free[hf], (uint32_t)(g - 1) & 1u, err);
            tc_fence_after();
            const uint64_t off = (uint64_t)((hf * QH * 128) >> 4);
            mma_hs_ss<Hs<HS>::KS>(tSt + hf * QH, dK, 128, dQ + off, QS, idS);
            mma_hs_ss<Hs<HS>::KS>(tdPt + hf * QH, dV, 128, dD + off, QS, idS);
            if (hf == 1 && j == nsub - 1) tc_commit(&kv_empty[kvb]);
            tc_commit(&s_full[hf]);
          }
        }
      }
    }
  } else if (warp == KV_CW + 2) {
    // ---------------------------------------------------------------- gradient MMAs
    // dV, dK (g, half) once P^T, dS^T of the half are in TMEM; a thread on
    // another scheduler than the score MMAs' issuer
    if (lane == 0) {
      const uint32_t idO = tc_idesc_bf16(128, HS, false, true);
      int g = 0;
      for (int r = 0;; r++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int k0 = (idx / BH) * 128;
        const int nsub = (T - k0 + QS - 1) / QS;
        for (int j = 0; j < nsub; j++, g++) {
          const int s = g % ST;
          const uint64_t dQn = ndesc(smem_u32(sQ + s * QTILE), QS, 0), dDn = ndesc(smem_u32(sD + s * QTILE), QS, 0);
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            mbar_wait(&p_full[hf], (uint32_t)g & 1u, err);
            tc_fence_after();
            // K = the half's QH queries: P^T / dS^T columns hf*QH/2.., q / dy rows hf*QH..
            mma_ts_chain<QH / 16>(tdV, tPt + hf * (QH / 2), dDn + nstep(hf * (QH / 16)), idO, j > 0 || hf > 0);
            mma_ts_chain<QH / 16>(tdK, tdSt + hf * (QH / 2), dQn + nstep(hf * (QH / 16)), idO, j > 0 || hf > 0);
            tc_commit(&p_empty[hf]);
            if (hf == 1) tc_commit(&q_empty[s]);
            if (hf == 1 && j == nsub - 1) tc_commit(acc_full);
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- elementwise warps
    const int quarter = warp & 3, cg = warp >> 2, grp = cg >> 1;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    // epilogue of an item, by group 0 (warps 0..7): warps with cg 0 take
    // dV, cg 1 dK, all HS columns of their 32 key rows.  It runs one item
    // late: epi_load reads the accumulators (everything that must precede
    // the next item's first gradient products, which wait for group 0),
    // epi_rest writes them out.
    constexpr int EH = HS;
    const int which = cg & 1;  // 0 dV, 1 dK
    const float mul = which ? scale : 1.f;
    struct Item { int b, h, kb, k0; };
    Item pv = {0, 0, 0, 0};
    auto epi_load = [&](const Item& p) {
      if constexpr (Cf::STAGE_OUT) {
        // the warp's 32 key rows x 64 columns into the 128B-swizzled staging
        // tile of dV (cg 0) or dK (cg 1), once the previous item's stores
        // have read the staging area
        if (tid == 0) bulk_wait_read0();
        named_bar_sync(1, KV_GW * 32);
        uint8_t* rowp = sOut + which * 16384 + row * 128;
#pragma unroll
        for (int e = 0; e < 2; e++) {
          uint32_t ra[32];
          tmem_ld32((which ? tdK : tdV) + lb + e * 32, ra);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; q++) {
            uint4 u;
            u.x = pack_bf16(__uint_as_float(ra[8 * q]) * mul, __uint_as_float(ra[8 * q + 1]) * mul);
            u.y = pack_bf16(__uint_as_float(ra[8 * q + 2]) * mul, __uint_as_float(ra[8 * q + 3]) * mul);
            u.z = pack_bf16(__uint_as_float(ra[8 * q + 4]) * mul, __uint_as_float(ra[8 * q + 5]) * mul);
            u.w = pack_bf16(__uint_as_float(ra[8 * q + 6]) * mul, __uint_as_float(ra[8 * q + 7]) * mul);
            *reinterpret_cast<uint4*>(rowp + (((4 * e + q) ^ (row & 7)) << 4)) = u;
          }
        }
      } else {
        // rows straight to global memory
        constexpr int EC = EH < 32 ? EH : 32;  // columns per chunk
        const int64_t C3 = 3 * (int64_t)C;
#pragma unroll
        for (int e = 0; e < EH; e += EC) {
          uint32_t rc[EC];
          tmem_ld_cols<EC>((which ? tdK : tdV) + lb + e, rc);
          tmem_ld_wait();
          float v[EC];
#pragma unroll
          for (int i = 0; i < EC; i++) v[i] = __uint_as_float(rc[i]);
          if (p.k0 + row < T)
            store_bf16_row<EC>(dqkv + ((int64_t)p.b * T + p.k0 + row) * C3 + (which ? C : 2 * C) + p.h * HS + e, v, mul);
        }
      }
    };
    auto epi_rest = [&](const Item& p) {
      if constexpr (Cf::STAGE_OUT) {
        // one thread stores the dV and dK tiles with TMA (rows past T are
        // not written)
        fence_proxy_async_smem();
        named_bar_sync(1, KV_GW * 32);
        if (tid == 0) {
          tma_store_3d(&tm_out, sOut, 2 * C + p.h * HS, p.k0, p.b);        // dV
          tma_store_3d(&tm_out, sOut + 16384, C + p.h * HS, p.k0, p.b);    // dK
          bulk_commit();
        }
        // the tiles' column sums over the block's key rows below T (one
        // partial row of the qkv bias gradient per (batch row, key block)),
        // read back from the staging tiles: warp w sums 32 rows of tile
        // w / 4, lane l columns 2l and 2l + 1; the 4 row groups are then
        // added in order
        const int tt = warp >> 2, rg = warp & 3, c2 = 2 * lane;
        const float2 cs = tile_colsum2<32>(sOut + tt * 16384, rg * 32, T - p.k0, lane);
        red[(tt * 4 + rg) * 64 + c2] = cs.x;
        red[(tt * 4 + rg) * 64 + c2 + 1] = cs.y;
        named_bar_sync(1, KV_GW * 32);
        if (tid < 128) {
          const int t2 = tid >> 6, col = tid & 63;
          float sum = 0.f;
#pragma unroll
          for (int q = 0; q < 4; q++) sum += red[(t2 * 4 + q) * 64 + col];
          bias_partial[((int64_t)p.b * nkb + p.kb) * 3 * (int64_t)C + (t2 ? C : 2 * C) + p.h * HS + col] = sum;
        }
      }
    };
    int g = 0, it = 0;
    for (int r = 0;; r++, it++) {
      const int idx = snake_item(r);
      if (idx >= nitems) break;
      const int kb = idx / BH, bh = idx % BH, b = bh / NH, h = bh % NH, k0 = kb * 128;
      const int key = k0 + row;
      const int nsub = (T - k0 + QS - 1) / QS;
      for (int j = 0; j < nsub; j++, g++) {
        const int s = g % ST, q0 = k0 + j * QS;
        mbar_wait(&s_full[grp], (uint32_t)g & 1u, err);
        tc_fence_after();
        const int c0 = q0 + cg * CPT;  // query of column 0 of this warp
        const float* lc = sLD + s * 2 * QS + cg * CPT;  // minus lse, minus D of the columns
        const bool edge = q0 < k0 + 128 || q0 + QS > T;
        // two halves of HC columns, each loaded, computed and stored before
        // the next is loaded (the TMEM loads and stores keep the order), so
        // that one half's operands and results are live at a time; the
        // group's S^T and dP^T columns are free once both halves are read
        constexpr int HC = CPT / 2;
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          uint32_t rs[HC], rd[HC];
          tmem_ld_cols<HC>(tSt + lb + cg * CPT + hh * HC, rs);
          tmem_ld_cols<HC>(tdPt + lb + cg * CPT + hh * HC, rd);
          tmem_ld_wait();
          if (hh == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[grp]);
          } else if (staged) {
            mbar_wait(&q_full[s], (uint32_t)(g / ST) & 1u, err);  // the stage's lse / D
          }
          uint32_t pk[HC / 2], dk[HC / 2];
          const float *gl = lse + (int64_t)bh * T, *gd = dsum + (int64_t)bh * T;
          if (staged) {
            if (edge)
              kv_elementwise<HC, true, true>(rs, rd, lc + hh * HC, lc + QS + hh * HC, gl, gd, c0 + hh * HC, key, T, sl2, pk, dk);
            else
              kv_elementwise<HC, false, true>(rs, rd, lc + hh * HC, lc + QS + hh * HC, gl, gd, c0 + hh * HC, key, T, sl2, pk, dk);
          } else {
            if (edge)
              kv_elementwise<HC, true, false>(rs, rd, lc + hh * HC, lc + QS + hh * HC, gl, gd, c0 + hh * HC, key, T, sl2, pk, dk);
            else
              kv_elementwise<HC, false, false>(rs, rd, lc + hh * HC, lc + QS + hh * HC, gl, gd, c0 + hh * HC, key, T, sl2, pk, dk);
          }
          if (hh == 0 && g > 0) {
            mbar_wait(&p_empty[grp], (uint32_t)(g - 1) & 1u, err);  // dV, dK(g-1) have read the half's P^T, dS^T
            tc_fence_after();
          }
          tmem_st_cols<HC / 2>(tPt + lb + cg * (CPT / 2) + hh * (HC / 2), pk);
          tmem_st_cols<HC / 2>(tdSt + lb + cg * (CPT / 2) + hh * (HC / 2), dk);
        }
        tmem_st_wait();
        const bool epi = grp == 0 && j == 0 && it > 0;
        if (epi) {
          // the previous item's dV, dK leave TMEM before this item's first
          // gradient products (half 0, group 0's) overwrite them; the rest
          // of its epilogue runs while the tensor pipe works on this item
          mbar_wait(acc_full, (uint32_t)(it - 1) & 1u, err);
          tc_fence_after();
          epi_load(pv);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[grp]);
        if (epi) epi_rest(pv);
      }
      pv = Item{b, h, kb, k0};
    }
    if (grp == 0 && it > 0) {  // the last item's epilogue
      mbar_wait(acc_full, (uint32_t)(it - 1) & 1u, err);
      tc_fence_after();
      epi_load(pv);
      epi_rest(pv);
    }
  }
  if (Cf::STAGE_OUT && tid == 0) bulk_wait0();  // the last item's stores are complete
  tc_fence_before();
  __syncthreads();
  if (warp == KV_CW) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

// ============================================================ backward: dQ
// Item (128-query block, b*h), 128-key blocks, each taken in two column
// halves of 64 keys.  Warps 0..15 elementwise in two groups: group h (warps
// 8h..8h+7) owns key half h of every block (warps w and w+4 of a group share
// lane quarter w % 4 = 32 query rows and take 32 key columns each); warp 16
// issues the score products, warp 17 loads, warp 18 issues the dQ products.
//   S = q k^T, dP = dy v^T (M = 128 queries, N = 64 keys per half, K = HS);
//   dS = P (dP - D) into TMEM; dQ += dS k (N = HS, K = 64 keys per half).
// Each half has its own hand-offs, so one group's TMEM traffic and
// arithmetic overlap the other's and the tensor pipe; the item's epilogue
// is group 0's, one item late.
// TMEM: S 0..127, dP 128..255, dS 256..319, dQ 320..320+HS-1.
// smem: q, dy [QB] | K ring [KST] | V ring [VST] | barriers.
#define DQ_CW 16
#define DQ_GW 8  // warps per elementwise group
#define DQ_THREADS (DQ_CW * 32 + 96)
// The elementwise step of one query row over N key columns (c0 .. c0+N-1):
// dS = 2^(S sl2 - lse2) (dP - D), packed to bf16 pairs; nl2, nd2: minus
// lse2 and minus D of the row, paired.  MASK (the diagonal block): keys past
// the query give 0.  A separate instantiation, so that blocks off the
// diagonal carry no compare-and-select per element.
template <int N, bool MASK>
__device__ __forceinline__ void dq_elementwise(const uint32_t* rs, const uint32_t* rd, uint64_t sl2x2, uint64_t nl2,
                                               uint64_t nd2, int c0, int q, uint32_t* dk) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[i]), __uint_as_float(rs[i + 1])), sl2x2, nl2), x0, x1);
    const float p0 = ex2_hw(x0), p1 = ex2_hw(x1);
    float d0, d1;
    f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(__uint_as_float(rd[i]), __uint_as_float(rd[i + 1])), nd2)), d0, d1);
    if (MASK) {
      d0 = c0 + i <= q ? d0 : 0.f;
      d1 = c0 + i + 1 <= q ? d1 : 0.f;
    }
    dk[i >> 1] = pack_bf16(d0, d1);
  }
}

template <int HS>
struct DqCfg {
  static constexpr uint32_t TILE = Hs<HS>::NB * 16384u;
  static constexpr int QB = HS > 64 ? 1 : 2;
  // a key stage is refilled only once dQ of its block has read it, so the
  // ring must cover the load latency past that point
  static constexpr int KST = HS > 64 ? 2 : 5;
  static constexpr int VST = HS > 64 ? 2 : 3;
  // head size 64: the dQ tile leaves through shared memory and one TMA store
  static constexpr bool STAGE_OUT = HS == 64;
  static constexpr uint32_t OUT_BYTES = STAGE_OUT ? 16384u : 0u;
  static constexpr uint32_t RED_BYTES = STAGE_OUT ? 8 * 64 * 4 : 0u;  // column-sum partials [8][64]
  static constexpr uint32_t SMEM = 1024 + QB * 2 * TILE + (KST + VST) * TILE + OUT_BYTES + RED_BYTES + 256;
};

template <int HS>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_dy,
                          const __grid_constant__ CUtensorMap tm_out, bf16* dqkv, const float* lse, const float* dsum,
                          float* bias_partial, int B, int T, int C, int NH, float scale, int* err) {
  using Cf = DqCfg<HS>;
  constexpr int QB = Cf::QB, KST = Cf::KST, VST = Cf::VST;
  constexpr uint32_t TILE = Cf::TILE;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sQ = sm;                     // [QB] x (q, dy)
  uint8_t* sK = sQ + QB * 2 * TILE;     // [KST]
  uint8_t* sV = sK + KST * TILE;        // [VST]
  uint8_t* sOut = sV + VST * TILE;  // dQ staging (head size 64)
  float* red = reinterpret_cast<float*>(sOut + Cf::OUT_BYTES);  // [8][64] column-sum partials
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + Cf::RED_BYTES);
  uint64_t* qd_full = bars;             // [QB]
  uint64_t* qd_empty = qd_full + QB;    // [QB]: the item's last S, dP have read q, dy
  uint64_t* k_full = qd_empty + QB;     // [KST]
  uint64_t* k_empty = k_full + KST;     // [KST]: dQ of the block has read k
  uint64_t* v_full = k_empty + KST;     // [VST]
  uint64_t* v_empty = v_full + VST;     // [VST]
  uint64_t* s_full = v_empty + VST;     // [2] S, dP of a half in TMEM
  uint64_t* s_free = s_full + 2;        // [2] copied out by the half's group
  uint64_t* p_full = s_free + 2;        // [2] dS of a half written by its group
  uint64_t* ds_free = p_full + 2;       // [2] dQ of the block has read the half's dS
  uint64_t* dq_full = ds_free + 2;      // the item's dQ complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(dq_full + 1);

  const int nqb = (T + 127) / 128, BH = B * NH, nitems = nqb * BH;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < QB; i++) { mbar_init(&qd_full[i], 1); mbar_init(&qd_empty[i], 1); }
    for (int i = 0; i < KST; i++) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < VST; i++) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
    for (int i = 0; i < 2; i++) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], DQ_GW);
      mbar_init(&p_full[i], DQ_GW);
      mbar_init(&ds_free[i], 1);
    }
    mbar_init(dq_full, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_dy);
  }
  if (warp == DQ_CW) { tmem_alloc(tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  pdl_trigger();  // dependents launch only once every CTA holds its tensor memory
  pdl_wait();
  const uint32_t tS = tm, tdP = tm + 128, tdS = tm + 256, tdQ = tm + 320;

  if (warp == DQ_CW + 1) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      int g = 0, it = 0;
      for (int r = 0;; r++, it++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int qb = nqb - 1 - idx / BH, bh = idx % BH, b = bh / NH, h = bh % NH;
        const int ib = it % QB;
        if (it >= QB) mbar_wait(&qd_empty[ib], (uint32_t)(it / QB - 1) & 1u, err);
        mbar_arrive_expect_tx(&qd_full[ib], 2 * TILE);
        load_tile<HS>(sQ + ib * 2 * TILE, &tm_qkv, &qd_full[ib], h * HS, qb * 128, b, 128);
        load_tile<HS>(sQ + ib * 2 * TILE + TILE, &tm_dy, &qd_full[ib], h * HS, qb * 128, b, 128);
        for (int j = 0; j <= qb; j++, g++) {
          const int ks = g % KST, vs = g % VST;
          if (g >= KST) mbar_wait(&k_empty[ks], (uint32_t)(g / KST - 1) & 1u, err);
          mbar_arrive_expect_tx(&k_full[ks], TILE);
          load_tile<HS>(sK + ks * TILE, &tm_qkv, &k_full[ks], C + h * HS, j * 128, b, 128);
          if (g >= VST) mbar_wait(&v_empty[vs], (uint32_t)(g / VST - 1) & 1u, err);
          mbar_arrive_expect_tx(&v_full[vs], TILE);
          load_tile<HS>(sV + vs * TILE, &tm_qkv, &v_full[vs], 2 * C + h * HS, j * 128, b, 128);
        }
      }
    }
  } else if (warp == DQ_CW) {
    // ---------------------------------------------------------------- score MMAs
    if (lane == 0) {
      const uint32_t idS = tc_idesc_bf16(128, 64, false, false);
      int g = 0, it = 0;
      for (int r = 0;; r++, it++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int nk = nqb - idx / BH;
        const int ib = it % QB;
        mbar_wait(&qd_full[ib], (uint32_t)(it / QB) & 1u, err);
        const uint64_t dQ = kdesc(smem_u32(sQ + ib * 2 * TILE), 128, 0), dD = kdesc(smem_u32(sQ + ib * 2 * TILE + TILE), 128, 0);
        for (int j = 0; j < nk; j++, g++) {
          const int ks = g % KST, vs = g % VST;
          mbar_wait(&k_full[ks], (uint32_t)(g / KST) & 1u, err);
          mbar_wait(&v_full[vs], (uint32_t)(g / VST) & 1u, err);
          const uint64_t dK = kdesc(smem_u32(sK + ks * TILE), 128, 0), dV = kdesc(smem_u32(sV + vs * TILE), 128, 0);
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            // key half hf: rows 64 hf.. of the k / v tiles (8 KB in, a
            // multiple of the 1 KB swizzle atom)
            if (g > 0) mbar_wait(&s_free[hf], (uint32_t)(g - 1) & 1u, err);
            tc_fence_after();
            const uint64_t off = (uint64_t)((hf * 64 * 128) >> 4);
            mma_hs_ss<Hs<HS>::KS>(tS + hf * 64, dQ, 128, dK + off, 128, idS);
            mma_hs_ss<Hs<HS>::KS>(tdP + hf * 64, dD, 128, dV + off, 128, idS);
            if (hf == 1) {
              tc_commit(&v_empty[vs]);
              if (j == nk - 1) tc_commit(&qd_empty[ib]);
            }
            tc_commit(&s_full[hf]);
          }
        }
      }
    }
  } else if (warp == DQ_CW + 2) {
    // ---------------------------------------------------------------- dQ MMAs
    // dQ (+)= dS(g, half) k(g, half) once the half's dS is in TMEM, from a
    // thread on another scheduler than the score MMAs' issuer
    if (lane == 0) {
      const uint32_t idQ = tc_idesc_bf16(128, HS, false, true);
      int g = 0;
      for (int r = 0;; r++) {
        const int idx = snake_item(r);
        if (idx >= nitems) break;
        const int nk = nqb - idx / BH;
        for (int j = 0; j < nk; j++, g++) {
          const uint64_t dKn = ndesc(smem_u32(sK + (g % KST) * TILE), 128, 0);
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            mbar_wait(&p_full[hf], (uint32_t)g & 1u, err);
            tc_fence_after();
            // K = the half's 64 keys: dS columns 32 hf.., k rows 64 hf..
            mma_ts_chain<4>(tdQ, tdS + hf * 32, dKn + nstep(4 * hf), idQ, j > 0 || hf > 0);
            tc_commit(&ds_free[hf]);
            if (hf == 1) {
              tc_commit(&k_empty[g % KST]);
              if (j == nk - 1) tc_commit(dq_full);
            }
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- elementwise warps
    const int quarter = warp & 3, cg = warp >> 2, grp = cg >> 1;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const float sl2 = scale * LOG2E_F;
    // epilogue of an item, by group 0 (warps 0..7): warp cg (0 or 1) takes
    // dQ columns cg*HS/2 .. cg*HS/2 + HS/2 - 1 of its 32 query rows.  It runs
    // one item late: epi_load reads the accumulator (everything that must
    // precede the next item's first dQ products, which wait for group 0),
    // epi_rest writes it out.
    constexpr int EQ = HS / 2;
    struct Item { int b, h, qb; };
    Item pv = {0, 0, 0};
    auto epi_load = [&](const Item& p) {
      if constexpr (Cf::STAGE_OUT) {
        // 32 columns of the warp's 32 query rows into the 128B-swizzled
        // staging tile (row = query, 16-byte chunks 4cg .. 4cg+3), once the
        // previous item's store has read it
        if (tid == 0) bulk_wait_read0();
        named_bar_sync(1, DQ_GW * 32);
        uint32_t ra[32];
        tmem_ld32(tdQ + lb + cg * 32, ra);
        tmem_ld_wait();
        uint8_t* rowp = sOut + row * 128;
#pragma unroll
        for (int qq = 0; qq < 4; qq++) {
          uint4 u;
          u.x = pack_bf16(__uint_as_float(ra[8 * qq]) * scale, __uint_as_float(ra[8 * qq + 1]) * scale);
          u.y = pack_bf16(__uint_as_float(ra[8 * qq + 2]) * scale, __uint_as_float(ra[8 * qq + 3]) * scale);
          u.z = pack_bf16(__uint_as_float(ra[8 * qq + 4]) * scale, __uint_as_float(ra[8 * qq + 5]) * scale);
          u.w = pack_bf16(__uint_as_float(ra[8 * qq + 6]) * scale, __uint_as_float(ra[8 * qq + 7]) * scale);
          *reinterpret_cast<uint4*>(rowp + (((cg * 4 + qq) ^ (row & 7)) << 4)) = u;
        }
      } else {
        // rows straight to global memory
        const int q = p.qb * 128 + row;
        constexpr int EC = EQ < 32 ? EQ : 32;  // columns per chunk
#pragma unroll
        for (int e = 0; e < EQ; e += EC) {
          uint32_t ra[EC];
          tmem_ld_cols<EC>(tdQ + lb + cg * EQ + e, ra);
          tmem_ld_wait();
          float v[EC];
#pragma unroll
          for (int i = 0; i < EC; i++) v[i] = __uint_as_float(ra[i]) * scale;
          if (q < T) store_bf16_row<EC>(dqkv + ((int64_t)p.b * T + q) * 3 * (int64_t)C + p.h * HS + cg * EQ + e, v, 1.f);
        }
      }
    };
    auto epi_rest = [&](const Item& p) {
      if constexpr (Cf::STAGE_OUT) {
        // one TMA store of the [128 x 64] tile (rows past T are not written)
        fence_proxy_async_smem();
        named_bar_sync(1, DQ_GW * 32);
        if (tid == 0) {
          tma_store_3d(&tm_out, sOut, p.h * HS, p.qb * 128, p.b);
          bulk_commit();
        }
        // column sums of the tile over its query rows below T (one partial
        // row of the qkv bias gradient per (batch row, query block)): warp w
        // sums 16 rows, lane l columns 2l and 2l + 1, then the 8 row groups
        // are added in order
        const int c2 = 2 * lane;
        const float2 cs = tile_colsum2<16>(sOut, warp * 16, T - p.qb * 128, lane);
        red[warp * 64 + c2] = cs.x;
        red[warp * 64 + c2 + 1] = cs.y;
        named_bar_sync(1, DQ_GW * 32);
        if (tid < 64) {
          float sum = 0.f;
#pragma unroll
          for (int q = 0; q < 8; q++) sum += red[q * 64 + tid];
          bias_partial[((int64_t)p.b * nqb + p.qb) * 3 * (int64_t)C + p.h * HS + tid] = sum;
        }
      }
    };
    int g = 0, it = 0;
    for (int r = 0;; r++, it++) {
      const int idx = snake_item(r);
      if (idx >= nitems) break;
      const int qb = nqb - 1 - idx / BH, bh = idx % BH, b = bh / NH, h = bh % NH;
      const int q = qb * 128 + row, nk = qb + 1;
      // minus the row's lse (base 2) and minus its D; rows past T give P = 0
      const float nl = q < T ? lse[(int64_t)bh * T + q] : -INFINITY;
      const float nd = q < T ? dsum[(int64_t)bh * T + q] : 0.f;
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(nl, nl), nd2 = f2_pack(nd, nd);
      for (int j = 0; j < nk; j++, g++) {
        mbar_wait(&s_full[grp], (uint32_t)g & 1u, err);
        tc_fence_after();
        const bool diag = j == nk - 1;
        // two pieces of 16 columns, each loaded, computed and stored before
        // the next is loaded; the group's S and dP columns are free once
        // both pieces are read
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          uint32_t rs[16], rd[16];
          tmem_ld16(tS + lb + cg * 32 + hh * 16, rs);
          tmem_ld16(tdP + lb + cg * 32 + hh * 16, rd);
          tmem_ld_wait();
          if (hh == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[grp]);
          }
          const int c0 = j * 128 + cg * 32 + hh * 16;  // key of the piece's column 0
          uint32_t dk[8];
          if (diag)  // the block on the diagonal: keys past the query give 0
            dq_elementwise<16, true>(rs, rd, sl2x2, nl2, nd2, c0, q, dk);
          else
            dq_elementwise<16, false>(rs, rd, sl2x2, nl2, nd2, c0, q, dk);
          if (hh == 0 && g > 0) {
            mbar_wait(&ds_free[grp], (uint32_t)(g - 1) & 1u, err);  // dQ(g-1) has read the half's dS
            tc_fence_after();
          }
          tmem_st8(tdS + lb + cg * 16 + hh * 8, dk);
        }
        tmem_st_wait();
        const bool epi = grp == 0 && j == 0 && it > 0;
        if (epi) {
          // the previous item's dQ leaves TMEM before this item's first dQ
          // products (half 0, group 0's) overwrite it; the rest of its
          // epilogue runs while the tensor pipe works on this item
          mbar_wait(dq_full, (uint32_t)(it - 1) & 1u, err);
          tc_fence_after();
          epi_load(pv);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[grp]);
        if (epi) epi_rest(pv);
      }
      pv = Item{b, h, qb};
    }
    if (grp == 0 && it > 0) {  // the last item's epilogue
      mbar_wait(dq_full, (uint32_t)(it - 1) & 1u, err);
      tc_fence_after();
      epi_load(pv);
      epi_rest(pv);
    }
  }
  if (Cf::STAGE_OUT && tid == 0) bulk_wait0();  // the last item's store is complete
  tc_fence_before();
  __syncthreads();
  if (warp == DQ_CW) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

// ============================================================ launchers
template <int HS>
static void fwd_hs(LaunchCtx& c, bf16* y, float* lse, const bf16* qkv, int B, int T, int C, int NH) {
  using Cf = FwdCfg<HS>;
  CUtensorMap tq, ty;
  if (!make_tmap_btw(&tq, qkv, B, T, 3 * C, 128) || !make_tmap_btw(&ty, y, B, T, C, 128)) {
    c.host_fail = 1;
    return;
  }
  const int nitems = ((T + 127) / 128) * B * NH;
  const int grid = std::min(nitems, Cf::PER_SM * c.num_sms);
  cudaFuncSetAttribute(attn_fwd_tc_kernel<HS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::SMEM);
  launch_pdl(c, attn_fwd_tc_kernel<HS>, dim3(grid), dim3(FW_THREADS), Cf::SMEM, tq, ty, y, lse, B, T, C, NH,
             1.f / sqrtf((float)HS), c.err);
}

void launch_attention_fwd_bf16(LaunchCtx& c, bf16* y, float* lse, const bf16* qkv, int B, int T,
                               int C, int NH) {
  switch (C / NH) {  // head sizes 16, 32, 64, 128 (checked at build)
    case 16: fwd_hs<16>(c, y, lse, qkv, B, T, C, NH); break;
    case 32: fwd_hs<32>(c, y, lse, qkv, B, T, C, NH); break;
    case 64: fwd_hs<64>(c, y, lse, qkv, B, T, C, NH); break;
    case 128: fwd_hs<128>(c, y, lse, qkv, B, T, C, NH); break;
    default: c.host_fail = 1;
  }
}

template <int HS>
static void bwd_hs(LaunchCtx& c, bf16* dqkv, const bf16* dy, const bf16* y, const bf16* qkv, const float* lse,
                   float* dsum, bool dsum_ready, int B, int T, int C, int NH, float* bias_partial) {
  using Kv = KvCfg<HS>;
  using Dq = DqCfg<HS>;
  CUtensorMap tq, tq_s, td, td_s, tout;
  if (!make_tmap_btw(&tq, qkv, B, T, 3 * C, 128) || !make_tmap_btw(&td, dy, B, T, C, 128) ||
      !make_tmap_btw(&tq_s, qkv, B, T, 3 * C, Kv::QS) || !make_tmap_btw(&td_s, dy, B, T, C, Kv::QS) ||
      !make_tmap_btw(&tout, dqkv, B, T, 3 * C, 128)) {
    c.host_fail = 1;
    return;
  }
  if (!dsum_ready) {
    const int64_t chunks = (int64_t)B * T * (C / 8);
    launch_pdl(c, attn_bwd_dsum_kernel<HS>, dim3((int)std::min<int64_t>((chunks + 255) / 256, (int64_t)c.num_sms * 8)),
               dim3(256), 0, dsum, dy, y, B, T, C, NH);
  }
  const float scale = 1.f / sqrtf((float)HS);
  const int nitems = ((T + 127) / 128) * B * NH;
  const int grid = std::min(nitems, c.num_sms);
  auto kv = (T & 3) == 0 ? attn_bwd_dkv_tc_kernel<HS, true> : attn_bwd_dkv_tc_kernel<HS, false>;
  cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Kv::SMEM);
  launch_pdl(c, kv, dim3(grid), dim3(KV_THREADS), Kv::SMEM, tq_s, tq, td_s, tout, dqkv, lse,
             (const float*)dsum, bias_partial, B, T, C, NH, scale, c.err);
  cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<HS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Dq::SMEM);
  launch_pdl(c, attn_bwd_dq_tc_kernel<HS>, dim3(grid), dim3(DQ_THREADS), Dq::SMEM, tq, td, tout, dqkv, lse,
             (const float*)dsum, bias_partial, B, T, C, NH, scale, c.err);
}

bool launch_attention_bwd_bf16(LaunchCtx& c, bf16* dqkv, const bf16* dy, const bf16* y,
                               const bf16* qkv, const float* lse, float* dsum, bool dsum_ready, int B, int T,
                               int C, int NH, float* bias_partial) {
  switch (C / NH) {
    case 16: bwd_hs<16>(c, dqkv, dy, y, qkv, lse, dsum, dsum_ready, B, T, C, NH, bias_partial); return false;
    case 32: bwd_hs<32>(c, dqkv, dy, y, qkv, lse, dsum, dsum_ready, B, T, C, NH, bias_partial); return false;
    case 64: bwd_hs<64>(c, dqkv, dy, y, qkv, lse, dsum, dsum_ready, B, T, C, NH, bias_partial); return true;
    case 128: bwd_hs<128>(c, dqkv, dy, y, qkv, lse, dsum, dsum_ready, B, T, C, NH, bias_partial); return false;
    default: c.host_fail = 1; return false;
  }
}
