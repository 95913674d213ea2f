// kernels.h -- host-side launchers of every kernel in libgpt2.so.
//
// Each launcher takes raw device pointers, sizes and a LaunchCtx (stream,
// device error word, launch counter) and enqueues its kernel(s); none
// allocates memory or synchronises.  Scratch buffers are passed in by the
// caller (the model owns them).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

struct LaunchCtx {
  cudaStream_t stream;
  int* err;           // device error word (DEVERR_* bits)
  int64_t* launches;  // host-side count of kernel launches
  int num_sms;
  int host_fail;      // set by a launcher that could not enqueue its kernel
  int pdl = 1;        // 0: launch_pdl launches without programmatic serialisation,
                      // so the first kernel waits for all earlier work on the stream
};

// Launch kernel `k` on c.stream with programmatic stream serialisation
// (the kernel calls pdl_trigger / pdl_wait, common.cuh) and count it.
template <typename... KArgs, typename... Args>
inline void launch_pdl(LaunchCtx& c, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = c.pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...) != cudaSuccess) c.host_fail = 1;
  (*c.launches)++;
}

// Same, with thread-block clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
inline void launch_pdl_cluster(LaunchCtx& c, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = cluster_x;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...) != cudaSuccess) c.host_fail = 1;
  (*c.launches)++;
}

// ---------------------------------------------------------------- init
struct InitSpec {
  int64_t off[17];  // start of each of the 16 parameter tensors, off[16] = total
  int L, C, V;
  uint64_t seed;
};
void launch_init_params(LaunchCtx& c, float* params, const InitSpec& s);
void launch_f32_to_bf16(LaunchCtx& c, bf16* out, const float* in, int64_t n);

// ---------------------------------------------------------------- encoder
// out[b,t,:] = wte[tok[b,t],:] + wpe[t,:]; ids outside [0,V) set DEVERR_TOKEN
// and read row 0 instead.
void launch_encoder_fwd(LaunchCtx& c, float* out, const int32_t* tok, const float* wte,
                        const float* wpe, int B, int T, int C, int V);
// dwte[tok[i]] += dout[i], dwpe[t] += sum_b dout[b,t]; deterministic.
// scratch: keys (uint32 [M]), piece partials (float [M*C]).
void launch_encoder_bwd(LaunchCtx& c, float* dwte, float* dwpe, const float* dout,
                        const int32_t* tok, int B, int T, int C, int Vp, uint32_t* sorted,
                        float* partial);

// ---------------------------------------------------------------- LayerNorm
template <typename OutT>
void launch_layernorm_fwd(LaunchCtx& c, OutT* out, float* mean, float* rstd, const float* inp,
                          const float* w, const float* b, int N, int C);
// dres (+)= dx; dres_act = dres in ActT (if non-null); dw, db += column
// sums; dres_colsum (if non-null) += column sums of the updated dres; via
// partials (float [ln_partial_floats(N, C)]).  dy (the gradient of the
// LayerNorm output) is in ActT too.
template <typename ActT>
void launch_layernorm_bwd(LaunchCtx& c, float* dres, ActT* dres_act, float* dw, float* db,
                          float* dres_colsum, const ActT* dy, const float* inp, const float* w,
                          const float* mean, const float* rstd, int N, int C, bool accumulate,
                          float* partial);
int64_t ln_partial_floats(int N, int C);

// ---------------------------------------------------------------- column sums
// Floats of the partial rows launch_colsum_partials writes for an M x N matrix.
int64_t colsum_partial_floats(int M, int N);

// ---------------------------------------------------------------- deferred column reductions
// One reduction of partial rows: sum the nb rows of width W (row stride W)
// of `partial`, rows in a fixed order, and add columns [i*seg, (i+1)*seg)
// into d[i] (a null d[i] is skipped).  first_block: the job's first block
// in a launch of several jobs (ascending over the job list).
struct ReduceJob {
  float* d[3];
  const float* partial;
  int nb, W, seg, first_block;
};
int reduce_job_blocks(int W);
// Every job of a device-resident list in one launch of `blocks` blocks (the
// sum of reduce_job_blocks over the jobs); each job's sums are the same, bit
// for bit, as those of one reduction launch per job (the allocation-free
// LayerNorm backward's).
void launch_reduce_jobs(LaunchCtx& c, const ReduceJob* jobs, int njobs, int blocks);
// The LayerNorm backward (as launch_layernorm_bwd) without its reduction:
// writes its partial rows and returns their number (the job is the
// caller's: W = 3C, seg = C, d = {dw, db, dres_colsum}).
template <typename ActT>
int launch_layernorm_bwd_partials(LaunchCtx& c, float* dres, ActT* dres_act, const ActT* dy, const float* inp,
                                  const float* w, const float* mean, const float* rstd, int N, int C,
                                  bool accumulate, float* partial);
// Column sums of x [M x N] (row stride ld) as R = colsum_partial_floats(M, N)
// / N partial rows: row r sums the r-th of R contiguous chunks of x's rows
// (a fixed order); returns R.  A ReduceJob adds the rows up.
template <typename T>
int launch_colsum_partials(LaunchCtx& c, float* partial, const T* x, int M, int N, int64_t ld);

// ---------------------------------------------------------------- softmax + CE
// Per row i < M of logits [M, Vp]: loss_i = logsumexp(l[0:V]) - l[target];
// if dlogits: logits row <- (softmax - onehot(target)) * dscale (pad cols 0).
template <typename T>
void launch_crossentropy(LaunchCtx& c, T* logits, float* losses, const int32_t* targets, int M,
                         int V, int Vp, float dscale, bool dlogits);
// out[0] = mean of losses[0:M] (fixed-order reduction)
void launch_mean(LaunchCtx& c, float* out, const float* losses, int M);

// ---------------------------------------------------------------- AdamW
void launch_adamw(LaunchCtx& c, float* p, const float* g, float* m, float* v, bf16* shadow,
                  int64_t n, float lr, float b1, float b2, float eps, float wd, float c1,
                  float c2);

// ---------------------------------------------------------------- GEMM
// out[m, n] = sum_k A(m,k) * B(n,k) with
//   A(m,k) = A[m*lda + k] (a_kmajor) or A[k*lda + m] (M-major)
//   B(n,k) = B[n*ldb + k] (b_kmajor) or B[k*ldb + n] (N-major)
enum GemmEpi {
  EPI_STORE = 0,     // out = acc (+ bias)                          out: act or f32
  EPI_GELU_FWD,      // x = acc + bias: out = gelu'(x), out2 = gelu(x)       both act
  EPI_RESIDUAL,      // out(f32) = aux(f32) + acc + bias
  EPI_MUL_AUX,       // out(act) = acc * aux(act)  (the GELU backward with aux = gelu')
  EPI_ACCUM,         // out(f32) += acc
  EPI_DOT_AUX,       // out(act) = acc; per row and 64-column group (an attention
                     // head): dot_out = -sum(out * aux), out as rounded to act
};
struct GemmArgs {
  int M, N, K;
  const void* A; int64_t lda; bool a_kmajor;
  const void* B; int64_t ldb; bool b_kmajor;
  int epi;
  void* out; int64_t ldo; bool out_f32;
  const float* bias;  // [N] or null
  void* out2;         // EPI_GELU_FWD
  const void* aux;    // EPI_RESIDUAL (f32, ldo) / EPI_MUL_AUX (act, ldo)
  float* splitk_scratch;  // EPI_ACCUM with split-K (tensor-core path)
  int64_t splitk_scratch_floats;
  // split-K reduced inside the GEMM kernel, in split order, when the tile
  // count needs no more flags than this (zero on entry, left zero on exit;
  // else the partial planes in splitk_scratch and a reduction kernel)
  int* splitk_flags;
  int64_t splitk_flag_count;
  // EPI_MUL_AUX on the tensor-core path: if set, also the column sums of
  // the stored (bf16) output over each 32-row block, [ceil(M/32)][N] floats
  // (a ReduceJob adds them up)
  float* colsum_out;
  // if set (few-row and CUDA-core kernels only): out and out2 start
  // (*out_row) * out_row_stride elements further, read on the device (the
  // cache row of a generation step, fixed launch arguments for CUDA graphs)
  const int* out_row;
  int64_t out_row_stride;
  // E4M3 operands (launch_gemm_fp8): the accumulator is divided by
  // (*dequant_a) * (*dequant_b), the operands' per-tensor scales (device)
  const float* dequant_a;
  const float* dequant_b;
  // EPI_DOT_AUX (act = bf16, N a multiple of 64): row m = b * dot_T + t and
  // column group h = n / 64 write dot_out[(b * (N / 64) + h) * dot_T + t]
  float* dot_out;
  int dot_T;
};
// E4M3 operands A [M, K], B [N, K] (uint8 codes, K-major, lda / ldb in
// bytes, multiples of 16), EPI_STORE only (bias allowed), dequant_a / _b set:
// the CTA-pair kernel with kind::f8f6f4 MMAs.
void launch_gemm_fp8(LaunchCtx& c, const GemmArgs& g);
// E4M3 per-tensor quantisation of n values (fp32 or bf16): scale[1] (scratch,
// zeroed here) collects max|x|, scale[0] = s = 448 / max|x| (1 for all zeros),
// q[i] = E4M3(x[i] * s) rounded to nearest even, saturating.
void launch_fp8_quantize(LaunchCtx& c, const void* x, bool x_bf16, int64_t n, uint8_t* q, float* scale);
// fp32 operands, SIMT FFMA (no TF32)
void launch_gemm_f32(LaunchCtx& c, const GemmArgs& g);
// bf16 operands on tcgen05 tensor cores, fp32 accumulation in TMEM
void launch_gemm_bf16(LaunchCtx& c, const GemmArgs& g);
bool gemm_bf16_init();  // resolves the driver's tensor-map encoder; false on failure
// M <= 16 rows, both operands K-major, EPI_STORE / EPI_RESIDUAL / EPI_GELU_FWD:
// the generation-sized products (weights as the 128-row MMA operand, the few
// rows of A as N = 16; launch_gemm_bf16 uses it by itself for such arguments)
bool gemm_rows_applies(const GemmArgs& g);
void launch_gemm_rows(LaunchCtx& c, const GemmArgs& g);

// ---------------------------------------------------------------- attention
// qkv [B,T,3C] -> y [B,T,C], lse [B,NH,T]: the logsumexp of the scaled,
// masked scores of each query row, in natural-log units on the CUDA-core
// path (launch_attention_*_simt), and minus it in base-2 units (minus log2
// of the row's sum of 2^(score*scale*log2 e)) on the tensor-core path
// (*_bf16); each backward reads what its own forward wrote (the tensor-core
// backward also keeps D = rowsum(dy * y) negated in dsum).
template <typename T>
void launch_attention_fwd_simt(LaunchCtx& c, T* y, float* lse, const T* qkv, int B, int T_,
                               int C, int NH);
template <typename T>
void launch_attention_bwd_simt(LaunchCtx& c, T* dqkv, const T* dy, const T* y, const T* qkv,
                               const float* lse, float* dsum, int B, int T_, int C, int NH,
                               float* scratch);
int64_t attention_simt_scratch_floats(int B, int T_, int NH);
void launch_attention_fwd_bf16(LaunchCtx& c, bf16* y, float* lse, const bf16* qkv, int B, int T_,
                               int C, int NH);
// qkv, y, dy -> dqkv [B,T,3C] (dq | dk | dv); dsum [B,NH,T] holds minus
// D = rowsum(dy * y) per head: computed here unless dsum_ready (the matmul
// that produced dy wrote it, EPI_DOT_AUX).
// Returns true when it also wrote the qkv bias gradient's partial rows
// (head size 64): bias_partial [B * ceil(T/128)][3C], row b * ceil(T/128) +
// block (a ReduceJob adds them up).
bool launch_attention_bwd_bf16(LaunchCtx& c, bf16* dqkv, const bf16* dy, const bf16* y,
                               const bf16* qkv, const float* lse, float* dsum, bool dsum_ready, int B,
                               int T_, int C, int NH, float* bias_partial);

// A tensor map over a [B][T][W] bf16 tensor with box {64, rows, 1},
// 128-byte swizzle, rows past T read as 0 (false if the driver's encoder is
// unavailable).  CUtensorMap is opaque here: a 128-byte aligned 128-byte blob.
struct CUtensorMap_st;
bool attn_tmap_btw(CUtensorMap_st* m, const void* base, int B, int T, int W, int rows);

// ---------------------------------------------------------------- decode
// Generation with the key/value cache qkv [B, T_, 3C] (row t of sequence b:
// [q | k | v] of position t): y[b*ldy + h*hs + d] = the attention of the
// query of row pos over rows 0..pos (head h, natural-log softmax, fp32).
// pos: device int (the position, read by the kernel).
template <typename T>
void launch_attention_decode(LaunchCtx& c, T* y, int64_t ldy, const T* qkv, int B, int T_, int C, int NH,
                             const int* pos);
// next[b] = the token drawn from logits[b*ld + 0..V-1]: inverse-CDF sampling
// of softmax(l / *temperature) at the uniform u[b] (*temperature <= 0: the
// first index of the largest score); temperature: device float.
template <typename T>
void launch_sample(LaunchCtx& c, int32_t* next, const T* logits, int64_t ld, int B, int V, const float* temperature,
                   const float* u);
// x[b, :] = wte[tok[b], :] + wpe[*pos, :] (ids outside [0, V) set
// DEVERR_TOKEN and read row 0)
void launch_decode_embed(LaunchCtx& c, float* x, const int32_t* tok, const float* wte, const float* wpe,
                         const int* pos, int B, int C, int V);
// the step's inputs into the model's buffers: tok_dst = tok_src, u_dst =
// u_src ([B] each), *pos_dst = pos, *temp_dst = temperature
void launch_decode_inputs(LaunchCtx& c, int32_t* tok_dst, const int32_t* tok_src, float* u_dst, const float* u_src,
                          int* pos_dst, int pos, float* temp_dst, float temperature, int B);

// One kernel whose mbarrier wait nothing completes: it gives up after the
// bounded-wait limit and sets DEVERR_TIMEOUT (tests of the error path).
void launch_expire_wait(LaunchCtx& c);

// Record the message gpt2_last_error(NULL) returns (entry points without a
// model handle).
void set_global_error(const char* msg);
