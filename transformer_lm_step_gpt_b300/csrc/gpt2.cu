// gpt2.cu -- the model object, its single device allocation, the step's
// launch sequence, and the C ABI declared in include/gpt2.h.
//
// Memory (QbitAI, section "Manually implementing each layer's forward/
// backward pass": everything is allocated once, as one 1-D block, and
// pointers are carved out of it): one cudaMalloc at build time holds the
// fp32 parameter / gradient / AdamW m / AdamW v arrays (same layout), the
// bf16 copy of the weights, every saved activation of every layer and the
// backward's scratch.  Nothing is allocated or freed afterwards.
//
// The step (InfoQ's layer list; GeekNews, "The Transformer core" for the
// block order):
//   forward   encoder -> L x [LN1 -> QKV -> attention -> proj + residual ->
//             LN2 -> fc + GELU -> fcproj + residual] -> LN_f -> tied head ->
//             softmax cross-entropy (dlogits computed in the same pass)
//   backward  head dgrad/wgrad -> LN_f -> L x reversed block -> encoder
//   update    one fused AdamW pass over the whole parameter array
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gpt2.h"
#include "common.cuh"
#include "kernels.h"

namespace {

enum { WTE = 0, WPE, LN1W, LN1B, QKVW, QKVB, ATTPROJW, ATTPROJB, LN2W, LN2B, FCW, FCB,
       FCPROJW, FCPROJB, LNFW, LNFB, NT };
const char* kTensorNames[NT] = {"wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw",
                                "attprojb", "ln2w", "ln2b", "fcw", "fcb", "fcprojw",
                                "fcprojb", "lnfw", "lnfb"};

thread_local std::string g_build_error = "no error";

// Kernel classes timed by gpt2_profile_*; work unit per class.
// Matmul classes are per Linear (qkv, attproj, fc, fcproj, the tied head)
// and per pass (forward, data gradient, weight gradient).
enum GemmSite { GS_QKV = 0, GS_ATTPROJ, GS_FC, GS_FCPROJ, GS_HEAD, GS_N };
enum GemmPass { GP_FWD = 0, GP_DGRAD, GP_WGRAD };
enum ProfClass { PC_GEMM0 = 0, PC_ATTN_FWD = 3 * GS_N, PC_ATTN_BWD, PC_LN_FWD, PC_LN_BWD, PC_CE,
                 PC_BIAS_GRAD, PC_ENC_FWD, PC_ENC_BWD, PC_ADAMW, PC_ZERO_GRAD, PC_DEC_ATTN, PC_SAMPLE,
                 PC_N };
const char* kProfNames[PC_N] = {
    "gemm_qkv_fwd", "gemm_qkv_dgrad", "gemm_qkv_wgrad",
    "gemm_attproj_fwd", "gemm_attproj_dgrad", "gemm_attproj_wgrad",
    "gemm_fc_fwd", "gemm_fc_dgrad", "gemm_fc_wgrad",
    "gemm_fcproj_fwd", "gemm_fcproj_dgrad", "gemm_fcproj_wgrad",
    "gemm_head_fwd", "gemm_head_dgrad", "gemm_head_wgrad",
    "attention_fwd", "attention_bwd", "layernorm_fwd", "layernorm_bwd", "crossentropy",
    "bias_grad", "encoder_fwd", "encoder_bwd", "adamw", "zero_grad", "decode_attention", "sample"};
const char* kProfUnits[PC_N] = {
    "flop", "flop", "flop", "flop", "flop", "flop", "flop", "flop", "flop", "flop", "flop",
    "flop", "flop", "flop", "flop", "flop", "flop", "byte", "byte", "byte", "byte", "byte",
    "byte", "byte", "byte", "byte", "byte"};

struct ProfState {
  uint32_t mask = 0;
  int64_t launches[PC_N] = {};
  double work[PC_N] = {}, ms[PC_N] = {};
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> pending;
  std::vector<cudaEvent_t> pool;
};

struct Bump {
  char* base;
  size_t off = 0;
  explicit Bump(char* b) : base(b) {}
  template <typename T>
  T* take(size_t n) {
    off = (off + 255) & ~(size_t)255;
    T* p = reinterpret_cast<T*>(base + off);
    off += n * sizeof(T);
    return p;
  }
};

}  // namespace

struct gpt2_model {
  gpt2_config cfg;
  int L, C, NH, V, Vp, maxT, B, T, M;
  bool bf;      // bf16 mode
  size_t act;   // bytes per stored activation element (2 or 4)
  int device = 0, num_sms = 148;
  cudaStream_t stream = nullptr;
  int64_t n_params = 0;
  int64_t off[NT + 1];
  char* block = nullptr;
  size_t block_bytes = 0;
  // fp32 arrays sharing the parameter layout
  float *params, *grads, *adam_m, *adam_v;
  bf16* wb = nullptr;  // bf16 copy of the parameters (bf16 mode)
  // inputs of the last forward
  int32_t *tok, *tgt;
  // activations (act = bf16 or fp32 per mode; residual stream fp32)
  std::vector<float*> res;  // L+1 residual streams [M,C]; res[0] = encoder output
  std::vector<float*> mid;  // L after-attention residuals [M,C]
  char *ln1, *qkv, *atty, *ln2, *fcd, *fcg, *lnf, *logits;
  float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd, *lse, *lnf_mean, *lnf_rstd;
  float *losses, *loss;
  // backward scratch
  float* dres;
  char* dres_act;  // bf16 copy of dres (bf16 mode); == dres in fp32 mode
  float* dln;
  char *dbig, *datty;
  float *dsum, *splitk;
  int64_t splitk_floats;
  int* splitk_flags;  // turnstiles of the in-kernel split-K reduction
  int64_t splitk_flag_count;
  uint32_t* enc_sorted;
  float* enc_partial;
  // partial rows of the bias and LayerNorm weight gradients, one slot per
  // reduction of a backward pass, added up by one launch at its end
  float* red_part;
  ReduceJob* red_jobs_dev;  // the job list on the device
  int red_jobs_cap = 0;
  std::vector<ReduceJob> red_jobs, red_jobs_up;  // this pass's jobs / the list on the device
  int* err;
  int64_t launches = 0;
  ProfState prof;
  // generation: one row per sequence (the key/value cache is qkv above)
  float *dec_x, *dec_mid, *dec_mean, *dec_rstd;
  char *dec_ln, *dec_y, *dec_fcd, *dec_fcg, *dec_logits;
  int32_t *dec_tok, *dec_next;  // the step's input ids and drawn ids [B]
  float *dec_u, *dec_temp;      // the step's uniforms [B] and temperature
  int* dec_pos;                 // the step's position
  // the decode step as a CUDA graph (its launches do not depend on the step)
  cudaStream_t dec_cap = nullptr;
  cudaGraph_t dec_graph = nullptr;
  cudaGraphExec_t dec_exec = nullptr;
  int64_t dec_graph_launches = 0;
  bool have_fwd = false, fwd_targets = false;
  bool have_cache = false;  // qkv holds keys / values of the current weights
  bool have_dec = false;    // dec_logits holds a decode step's scores
  std::string last_error = "no error";

  int64_t tensor(int t) const { return off[t]; }
  float* P(int t) const { return params + off[t]; }
  float* G(int t) const { return grads + off[t]; }
  const void* W(int t) const {  // matmul operand copy of a weight
    return bf ? static_cast<const void*>(wb + off[t]) : static_cast<const void*>(params + off[t]);
  }
  template <typename X = char>
  X* A(char* base, int l, int64_t per) const {  // per-layer slice of an activation array
    return reinterpret_cast<X*>(base + (size_t)l * per * act);
  }
};

namespace {

cudaEvent_t take_event(gpt2_model* m) {
  if (!m->prof.pool.empty()) {
    cudaEvent_t e = m->prof.pool.back();
    m->prof.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Names the launches made in its scope with an NVTX range of the class (for
// profilers; without one attached the calls do nothing), and records an
// event pair around them when the class is selected, accounting the launch
// and its algorithmic work.
struct ProfScope {
  gpt2_model* m = nullptr;
  int cls;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;
  ProfScope(gpt2_model* mm, int c, double work) : cls(c) {
    nvtxRangePushA(kProfNames[c]);
    if (!(mm->prof.mask & (1u << c))) return;
    m = mm;
    e0 = take_event(m);
    e1 = take_event(m);
    cudaEventRecord(e0, m->stream);
    m->prof.launches[c]++;
    m->prof.work[c] += work;
  }
  ~ProfScope() {
    if (m) {
      cudaEventRecord(e1, m->stream);
      m->prof.pending.push_back({cls, {e0, e1}});
    }
    nvtxRangePop();
  }
};

int fail(gpt2_model* m, int code, const std::string& msg) {
  if (m) m->last_error = msg;
  else g_build_error = msg;
  return code;
}

int cuda_fail(gpt2_model* m, cudaError_t e, const char* where) {
  return fail(m, GPT2_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

LaunchCtx ctx(gpt2_model* m) {
  LaunchCtx c;
  c.stream = m->stream;
  c.err = m->err;
  c.launches = &m->launches;
  c.num_sms = m->num_sms;
  c.host_fail = 0;
  return c;
}

int after_launches(gpt2_model* m, LaunchCtx& c, const char* where) {
  if (c.host_fail) return fail(m, GPT2_ERR_CUDA, std::string(where) + ": a kernel could not be enqueued");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(m, e, where);
  return GPT2_OK;
}

// Read and clear the device error word (synchronises the stream first).
int check_device(gpt2_model* m, const char* where) {
  cudaError_t e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) return cuda_fail(m, e, where);
  int w = 0;
  e = cudaMemcpy(&w, m->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(m, e, where);
  if (w) {
    cudaMemset(m->err, 0, sizeof(int));
    // a launch that gave up may have left split-K turnstiles set
    if (m->splitk_flag_count) cudaMemset(m->splitk_flags, 0, sizeof(int) * m->splitk_flag_count);
    if (w & DEVERR_TIMEOUT) return fail(m, GPT2_ERR_TIMEOUT, std::string(where) + ": a bounded device wait expired");
    if (w & DEVERR_TOKEN) return fail(m, GPT2_ERR_TOKEN, std::string(where) + ": token or target id outside [0, V)");
  }
  return GPT2_OK;
}

void param_sizes(const gpt2_model* m, int64_t n[NT]) {
  const int64_t L = m->L, C = m->C;
  n[WTE] = (int64_t)m->Vp * C; n[WPE] = (int64_t)m->maxT * C;
  n[LN1W] = L * C; n[LN1B] = L * C; n[QKVW] = L * 3 * C * C; n[QKVB] = L * 3 * C;
  n[ATTPROJW] = L * C * C; n[ATTPROJB] = L * C; n[LN2W] = L * C; n[LN2B] = L * C;
  n[FCW] = L * 4 * C * C; n[FCB] = L * 4 * C; n[FCPROJW] = L * C * 4 * C; n[FCPROJB] = L * C;
  n[LNFW] = C; n[LNFB] = C;
}

// Carve every buffer out of one block (base == nullptr: measure only).
size_t layout(gpt2_model* m, char* base) {
  Bump b(base);
  const int64_t M = m->M, C = m->C, L = m->L, n = m->n_params;
  const size_t a = m->act;
  m->params = b.take<float>(n);
  m->grads = b.take<float>(n);
  m->adam_m = b.take<float>(n);
  m->adam_v = b.take<float>(n);
  m->wb = m->bf ? b.take<bf16>(n) : nullptr;
  m->tok = b.take<int32_t>(M);
  m->tgt = b.take<int32_t>(M);
  m->res.assign(L + 1, nullptr);
  m->mid.assign(L, nullptr);
  for (int l = 0; l <= L; l++) m->res[l] = b.take<float>(M * C);
  for (int l = 0; l < L; l++) m->mid[l] = b.take<float>(M * C);
  m->ln1 = b.take<char>(L * M * C * a);
  m->qkv = b.take<char>(L * M * 3 * C * a);
  m->atty = b.take<char>(L * M * C * a);
  m->ln2 = b.take<char>(L * M * C * a);
  m->fcd = b.take<char>(L * M * 4 * C * a);
  m->fcg = b.take<char>(L * M * 4 * C * a);
  m->lnf = b.take<char>(M * C * a);
  m->logits = b.take<char>(M * (int64_t)m->Vp * a);
  m->ln1_mean = b.take<float>(L * M);
  m->ln1_rstd = b.take<float>(L * M);
  m->ln2_mean = b.take<float>(L * M);
  m->ln2_rstd = b.take<float>(L * M);
  m->lse = b.take<float>(L * (int64_t)m->B * m->NH * m->T);
  m->lnf_mean = b.take<float>(M);
  m->lnf_rstd = b.take<float>(M);
  m->losses = b.take<float>(M);
  m->loss = b.take<float>(1);
  m->dres = b.take<float>(M * C);
  m->dres_act = m->bf ? b.take<char>(M * C * a) : reinterpret_cast<char*>(m->dres);
  m->dln = b.take<float>(M * C);
  m->dbig = b.take<char>(M * 4 * C * a);
  m->datty = b.take<char>(M * C * a);
  m->dsum = b.take<float>((int64_t)m->B * m->NH * m->T);
  m->splitk_floats = m->bf ? 16 * C * C : 0;
  m->splitk = b.take<float>(m->splitk_floats);
  m->splitk_flag_count = m->bf ? 8192 : 0;
  m->splitk_flags = b.take<int>(m->splitk_flag_count);
  m->enc_sorted = b.take<uint32_t>(M);
  m->enc_partial = b.take<float>(M * C);
  {
    // per layer: the LN2 and LN1 backward partials, the fc bias partials
    // (one row per 32 rows of the fcproj data gradient, or the column-sum
    // pass's rows) and the qkv bias partials (one row per batch row and
    // 128-query block from the attention backward, or the column-sum
    // pass's); and the final LayerNorm's
    const int64_t lnp = ln_partial_floats(m->M, m->C);
    const int64_t fcp = std::max<int64_t>((M + 31) / 32 * 4 * C, colsum_partial_floats(m->M, 4 * m->C));
    const int64_t qkvp = std::max<int64_t>((int64_t)m->B * ((m->T + 127) / 128) * 3 * C,
                                           colsum_partial_floats(m->M, 3 * m->C));
    m->red_part = b.take<float>(L * (2 * lnp + fcp + qkvp) + lnp + 64 * (4 * L + 1));  // + 256-byte slot alignment
    m->red_jobs_cap = 4 * m->L + 1;
    m->red_jobs_dev = b.take<ReduceJob>(m->red_jobs_cap);
  }
  m->dec_x = b.take<float>((int64_t)m->B * C);
  m->dec_mid = b.take<float>((int64_t)m->B * C);
  m->dec_mean = b.take<float>(m->B);
  m->dec_rstd = b.take<float>(m->B);
  m->dec_ln = b.take<char>((int64_t)m->B * C * a);
  m->dec_y = b.take<char>((int64_t)m->B * C * a);
  m->dec_fcd = b.take<char>((int64_t)m->B * 4 * C * a);
  m->dec_fcg = b.take<char>((int64_t)m->B * 4 * C * a);
  m->dec_logits = b.take<char>((int64_t)m->B * m->Vp * a);
  m->dec_tok = b.take<int32_t>(m->B);
  m->dec_next = b.take<int32_t>(m->B);
  m->dec_u = b.take<float>(m->B);
  m->dec_temp = b.take<float>(1);
  m->dec_pos = b.take<int>(1);
  m->err = b.take<int>(1);
  return b.off + 256;
}

GemmArgs gemm(int M, int N, int K, const void* A, int64_t lda, bool ak, const void* B,
              int64_t ldb, bool bk, int epi, void* out, int64_t ldo, bool out_f32) {
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.a_kmajor = ak;
  g.B = B; g.ldb = ldb; g.b_kmajor = bk;
  g.epi = epi; g.out = out; g.ldo = ldo; g.out_f32 = out_f32;
  return g;
}

void run_gemm(gpt2_model* m, LaunchCtx& c, GemmArgs g, int site) {
  const int pass = g.a_kmajor ? (g.b_kmajor ? GP_FWD : GP_DGRAD) : GP_WGRAD;
  ProfScope ps(m, PC_GEMM0 + 3 * site + pass, 2.0 * g.M * (double)g.N * g.K);
  if (m->bf) {
    g.splitk_scratch = m->splitk;
    g.splitk_scratch_floats = m->splitk_floats;
    g.splitk_flags = m->splitk_flags;
    g.splitk_flag_count = m->splitk_flag_count;
    launch_gemm_bf16(c, g);
  } else {
    launch_gemm_f32(c, g);
  }
}

template <typename ActT>
void forward_layers(gpt2_model* m, LaunchCtx& c, bool with_targets) {
  const int M = m->M, C = m->C, L = m->L, B = m->B, T = m->T, NH = m->NH;
  const bool f32 = !m->bf;
  const double a = (double)sizeof(ActT);
  const double attn_flop = 4.0 * B * NH * (double)(C / NH) * (T * (T + 1.0) / 2.0);
  {
    ProfScope ps(m, PC_ENC_FWD, 12.0 * M * C);
    launch_encoder_fwd(c, m->res[0], m->tok, m->P(WTE), m->P(WPE), B, T, C, m->V);
  }
  const int64_t WS = sizeof(ActT) == 2 ? 2 : 4;
  auto w = [&](int t, int64_t o) {
    return static_cast<const void*>(static_cast<const char*>(m->W(t)) + o * WS);
  };
  for (int l = 0; l < L; l++) {
    ActT* ln1 = m->A<ActT>(m->ln1, l, (int64_t)M * C);
    ActT* qkv = m->A<ActT>(m->qkv, l, (int64_t)M * 3 * C);
    ActT* atty = m->A<ActT>(m->atty, l, (int64_t)M * C);
    ActT* ln2 = m->A<ActT>(m->ln2, l, (int64_t)M * C);
    ActT* fcd = m->A<ActT>(m->fcd, l, (int64_t)M * 4 * C);
    ActT* fcg = m->A<ActT>(m->fcg, l, (int64_t)M * 4 * C);
    float* lse = m->lse + (int64_t)l * B * NH * T;
    {
      ProfScope ps(m, PC_LN_FWD, (double)M * C * (4 + a) + 8.0 * M);
      launch_layernorm_fwd<ActT>(c, ln1, m->ln1_mean + (int64_t)l * M, m->ln1_rstd + (int64_t)l * M,
                                 m->res[l], m->P(LN1W) + l * C, m->P(LN1B) + l * C, M, C);
    }
    GemmArgs g = gemm(M, 3 * C, C, ln1, C, true, w(QKVW, (int64_t)l * 3 * C * C), C, true,
                      EPI_STORE, qkv, 3 * C, f32);
    g.bias = m->P(QKVB) + (int64_t)l * 3 * C;
    run_gemm(m, c, g, GS_QKV);
    {
      ProfScope ps(m, PC_ATTN_FWD, attn_flop);
      if (f32) launch_attention_fwd_simt<ActT>(c, atty, lse, qkv, B, T, C, NH);
      else launch_attention_fwd_bf16(c, reinterpret_cast<bf16*>(atty), lse, reinterpret_cast<const bf16*>(qkv), B, T, C, NH);
    }
    g = gemm(M, C, C, atty, C, true, w(ATTPROJW, (int64_t)l * C * C), C, true, EPI_RESIDUAL,
             m->mid[l], C, true);
    g.bias = m->P(ATTPROJB) + (int64_t)l * C;
    g.aux = m->res[l];
    run_gemm(m, c, g, GS_ATTPROJ);
    {
      ProfScope ps(m, PC_LN_FWD, (double)M * C * (4 + a) + 8.0 * M);
      launch_layernorm_fwd<ActT>(c, ln2, m->ln2_mean + (int64_t)l * M, m->ln2_rstd + (int64_t)l * M,
                                 m->mid[l], m->P(LN2W) + l * C, m->P(LN2B) + l * C, M, C);
    }
    // fc: x = ln2 Wfc^T + b; fcg = gelu(x), and fcd = gelu'(x) for the backward
    g = gemm(M, 4 * C, C, ln2, C, true, w(FCW, (int64_t)l * 4 * C * C), C, true, EPI_GELU_FWD,
             fcd, 4 * C, f32);
    g.bias = m->P(FCB) + (int64_t)l * 4 * C;
    g.out2 = fcg;
    run_gemm(m, c, g, GS_FC);
    g = gemm(M, C, 4 * C, fcg, 4 * C, true, w(FCPROJW, (int64_t)l * C * 4 * C), 4 * C, true,
             EPI_RESIDUAL, m->res[l + 1], C, true);
    g.bias = m->P(FCPROJB) + (int64_t)l * C;
    g.aux = m->mid[l];
    run_gemm(m, c, g, GS_FCPROJ);
  }
  ActT* lnf = reinterpret_cast<ActT*>(m->lnf);
  {
    ProfScope ps(m, PC_LN_FWD, (double)M * C * (4 + a) + 8.0 * M);
    launch_layernorm_fwd<ActT>(c, lnf, m->lnf_mean, m->lnf_rstd, m->res[L], m->P(LNFW), m->P(LNFB), M, C);
  }
  ActT* logits = reinterpret_cast<ActT*>(m->logits);
  run_gemm(m, c, gemm(M, m->Vp, C, lnf, C, true, m->W(WTE), C, true, EPI_STORE, logits, m->Vp, f32), GS_HEAD);
  {
    ProfScope ps(m, PC_CE, (with_targets ? 2.0 : 1.0) * M * (double)m->Vp * a + 4.0 * M);
    launch_crossentropy<ActT>(c, logits, m->losses, with_targets ? m->tgt : nullptr, M, m->V, m->Vp,
                              1.f / (float)M, with_targets);
  }
  if (with_targets) launch_mean(c, m->loss, m->losses, M);
}

// One new position `pos` of every sequence with the key/value cache: the
// forward of forward_layers applied to row pos only (GeekNews, "A GPT-2-based
// ChatGPT clone in 3000 bytes of C", section "How KV caching works": the rows
// before it are reused, only the new one is computed).  Its k, v go into row
// pos of each layer's qkv; its attention reads rows 0..pos; the final
// LayerNorm output times wte^T gives the row's scores, from which the next
// token is drawn.
// Inputs in dec_tok, dec_pos, dec_temp, dec_u; the drawn ids go to
// dec_next.  dev_rows: the new cache row is located on the device (from
// dec_pos), so that the launches do not depend on the step (graph capture);
// otherwise at row `pos`.
template <typename ActT>
void decode_layers(gpt2_model* m, LaunchCtx& c, bool dev_rows, int pos) {
  const int M = m->M, C = m->C, L = m->L, B = m->B, T = m->T, NH = m->NH;
  const bool f32 = !m->bf;
  const int64_t WS = sizeof(ActT) == 2 ? 2 : 4;
  auto w = [&](int t, int64_t o) {
    return static_cast<const void*>(static_cast<const char*>(m->W(t)) + o * WS);
  };
  ActT* ln = reinterpret_cast<ActT*>(m->dec_ln);
  ActT* y = reinterpret_cast<ActT*>(m->dec_y);
  float *x = m->dec_x, *mid = m->dec_mid;
  const double a = (double)sizeof(ActT);
  const double ln_bytes = (double)B * C * (4 + a) + 8.0 * B;
  {
    ProfScope ps(m, PC_ENC_FWD, 12.0 * B * C);
    launch_decode_embed(c, x, m->dec_tok, m->P(WTE), m->P(WPE), m->dec_pos, B, C, m->V);
  }
  for (int l = 0; l < L; l++) {
    ActT* qkv = m->A<ActT>(m->qkv, l, (int64_t)M * 3 * C);
    {
      ProfScope ps(m, PC_LN_FWD, ln_bytes);
      launch_layernorm_fwd<ActT>(c, ln, m->dec_mean, m->dec_rstd, x, m->P(LN1W) + l * C, m->P(LN1B) + l * C, B, C);
    }
    // row pos of sequence b sits at qkv + (b*T + pos)*3C: rows of stride T*3C
    GemmArgs g = gemm(B, 3 * C, C, ln, C, true, w(QKVW, (int64_t)l * 3 * C * C), C, true, EPI_STORE,
                      dev_rows ? qkv : qkv + (int64_t)pos * 3 * C, (int64_t)T * 3 * C, f32);
    g.bias = m->P(QKVB) + (int64_t)l * 3 * C;
    if (dev_rows) {
      g.out_row = m->dec_pos;
      g.out_row_stride = 3 * (int64_t)C;
    }
    run_gemm(m, c, g, GS_QKV);
    {
      // the cached keys and values of rows 0..pos read once, the output row written
      ProfScope ps(m, PC_DEC_ATTN, a * ((double)B * (pos + 1) * 2 * C + 2.0 * B * C));
      launch_attention_decode<ActT>(c, y, C, qkv, B, T, C, NH, m->dec_pos);
    }
    g = gemm(B, C, C, y, C, true, w(ATTPROJW, (int64_t)l * C * C), C, true, EPI_RESIDUAL, mid, C, true);
    g.bias = m->P(ATTPROJB) + (int64_t)l * C;
    g.aux = x;
    run_gemm(m, c, g, GS_ATTPROJ);
    {
      ProfScope ps(m, PC_LN_FWD, ln_bytes);
      launch_layernorm_fwd<ActT>(c, ln, m->dec_mean, m->dec_rstd, mid, m->P(LN2W) + l * C, m->P(LN2B) + l * C, B, C);
    }
    g = gemm(B, 4 * C, C, ln, C, true, w(FCW, (int64_t)l * 4 * C * C), C, true, EPI_GELU_FWD, m->dec_fcd,
             4 * C, f32);
    g.bias = m->P(FCB) + (int64_t)l * 4 * C;
    g.out2 = m->dec_fcg;
    run_gemm(m, c, g, GS_FC);
    g = gemm(B, C, 4 * C, m->dec_fcg, 4 * C, true, w(FCPROJW, (int64_t)l * C * 4 * C), 4 * C, true,
             EPI_RESIDUAL, x, C, true);
    g.bias = m->P(FCPROJB) + (int64_t)l * C;
    g.aux = mid;
    run_gemm(m, c, g, GS_FCPROJ);
  }
  {
    ProfScope ps(m, PC_LN_FWD, ln_bytes);
    launch_layernorm_fwd<ActT>(c, ln, m->dec_mean, m->dec_rstd, x, m->P(LNFW), m->P(LNFB), B, C);
  }
  ActT* logits = reinterpret_cast<ActT*>(m->dec_logits);
  run_gemm(m, c, gemm(B, m->Vp, C, ln, C, true, m->W(WTE), C, true, EPI_STORE, logits, m->Vp, f32), GS_HEAD);
  {
    ProfScope ps(m, PC_SAMPLE, a * (double)B * m->V);
    launch_sample<ActT>(c, m->dec_next, logits, m->Vp, B, m->V, m->dec_temp, m->dec_u);
  }
}

template <typename ActT>
void backward_layers(gpt2_model* m, LaunchCtx& c) {
  const int M = m->M, C = m->C, L = m->L, B = m->B, T = m->T, NH = m->NH;
  const int Vp = m->Vp;
  const int64_t WS = sizeof(ActT) == 2 ? 2 : 4;
  auto w = [&](int t, int64_t o) {
    return static_cast<const void*>(static_cast<const char*>(m->W(t)) + o * WS);
  };
  const bool f32 = !m->bf;
  const double a = (double)sizeof(ActT);
  const double lnb_bytes = (double)M * C * (16.0 + (f32 ? 0.0 : a)) + 8.0 * M;
  const double attn_flop = 8.0 * B * NH * (double)(C / NH) * (T * (T + 1.0) / 2.0);
  ActT* dlogits = reinterpret_cast<ActT*>(m->logits);
  ActT* lnf = reinterpret_cast<ActT*>(m->lnf);
  ActT* dres_act = reinterpret_cast<ActT*>(m->dres_act);
  ActT* dres_act_out = f32 ? nullptr : dres_act;  // fp32 mode: dres itself is the operand
  ActT* dbig = reinterpret_cast<ActT*>(m->dbig);
  ActT* datty = reinterpret_cast<ActT*>(m->datty);
  // tied head: logits = lnf wte^T
  // the LayerNorm input gradients (dln) are in the activation type
  ActT* dln = reinterpret_cast<ActT*>(m->dln);
  // the bias and LayerNorm weight gradients are column sums: each kernel
  // that produces them leaves partial rows in a slot of its own, and one
  // launch at the end of the pass adds every slot up (the reductions feed
  // nothing inside the pass)
  float* slot = m->red_part;
  int red_blocks = 0;
  m->red_jobs.clear();
  auto take_slot = [&](int64_t floats) {
    float* p = slot;
    slot += (floats + 63) & ~(int64_t)63;
    return p;
  };
  auto add_job = [&](float* d0, float* d1, float* d2, const float* partial, int nb, int W, int seg) {
    ReduceJob j;
    j.d[0] = d0; j.d[1] = d1; j.d[2] = d2;
    j.partial = partial; j.nb = nb; j.W = W; j.seg = seg; j.first_block = red_blocks;
    red_blocks += reduce_job_blocks(W);
    m->red_jobs.push_back(j);
  };
  const int64_t lnp = ln_partial_floats(M, C);
  run_gemm(m, c, gemm(M, C, Vp, dlogits, Vp, true, m->W(WTE), C, false, EPI_STORE, dln, C, f32), GS_HEAD);
  run_gemm(m, c, gemm(Vp, C, M, dlogits, Vp, false, lnf, C, false, EPI_ACCUM, m->G(WTE), C, true), GS_HEAD);
  {
    ProfScope ps(m, PC_LN_BWD, lnb_bytes - 4.0 * M * C);
    float* part = take_slot(lnp);
    const int nb = launch_layernorm_bwd_partials<ActT>(c, m->dres, dres_act_out, dln, m->res[L], m->P(LNFW),
                                                       m->lnf_mean, m->lnf_rstd, M, C, false, part);
    add_job(m->G(LNFW), m->G(LNFB), m->G(FCPROJB) + (int64_t)(L - 1) * C, part, nb, 3 * C, C);
  }
  for (int l = L - 1; l >= 0; l--) {
    ActT* ln1 = m->A<ActT>(m->ln1, l, (int64_t)M * C);
    ActT* qkv = m->A<ActT>(m->qkv, l, (int64_t)M * 3 * C);
    ActT* atty = m->A<ActT>(m->atty, l, (int64_t)M * C);
    ActT* ln2 = m->A<ActT>(m->ln2, l, (int64_t)M * C);
    ActT* fcd = m->A<ActT>(m->fcd, l, (int64_t)M * 4 * C);
    ActT* fcg = m->A<ActT>(m->fcg, l, (int64_t)M * 4 * C);
    float* lse = m->lse + (int64_t)l * B * NH * T;
    // fcproj: res[l+1] = mid + fcg Wfcproj^T + b
    GemmArgs g = gemm(M, 4 * C, C, dres_act, C, true, w(FCPROJW, (int64_t)l * C * 4 * C), 4 * C,
                      false, EPI_MUL_AUX, dbig, 4 * C, f32);
    g.aux = fcd;  // d(fc pre-activation) = d(fcg) * gelu'(x)
    float* fcb_part = take_slot(std::max<int64_t>((int64_t)(M + 31) / 32 * 4 * C, colsum_partial_floats(M, 4 * C)));
    if (!f32) g.colsum_out = fcb_part;  // fc bias gradient partials, 32 rows each
    run_gemm(m, c, g, GS_FCPROJ);
    run_gemm(m, c, gemm(C, 4 * C, M, dres_act, C, false, fcg, 4 * C, false, EPI_ACCUM,
                        m->G(FCPROJW) + (int64_t)l * C * 4 * C, 4 * C, true), GS_FCPROJ);
    // fcproj bias gradient: column sums of dres, taken by the LayerNorm
    // backward that produced dres (LN_f or the next block's LN1)
    // fc: x = ln2 Wfc^T + b
    run_gemm(m, c, gemm(M, C, 4 * C, dbig, 4 * C, true, w(FCW, (int64_t)l * 4 * C * C), C, false,
                        EPI_STORE, dln, C, f32), GS_FC);
    run_gemm(m, c, gemm(4 * C, C, M, dbig, 4 * C, false, ln2, C, false, EPI_ACCUM,
                        m->G(FCW) + (int64_t)l * 4 * C * C, C, true), GS_FC);
    if (f32) {
      ProfScope ps(m, PC_BIAS_GRAD, a * M * 4.0 * C);
      const int nb = launch_colsum_partials<ActT>(c, fcb_part, dbig, M, 4 * C, 4 * C);
      add_job(m->G(FCB) + (int64_t)l * 4 * C, nullptr, nullptr, fcb_part, nb, 4 * C, 4 * C);
    } else {
      add_job(m->G(FCB) + (int64_t)l * 4 * C, nullptr, nullptr, fcb_part, (M + 31) / 32, 4 * C, 4 * C);
    }
    {
      ProfScope ps(m, PC_LN_BWD, lnb_bytes);
      float* part = take_slot(lnp);
      const int nb = launch_layernorm_bwd_partials<ActT>(c, m->dres, dres_act_out, dln, m->mid[l], m->P(LN2W) + l * C,
                                                         m->ln2_mean + (int64_t)l * M, m->ln2_rstd + (int64_t)l * M,
                                                         M, C, true, part);
      add_job(m->G(LN2W) + l * C, m->G(LN2B) + l * C, m->G(ATTPROJB) + (int64_t)l * C, part, nb, 3 * C, C);
    }
    // attproj: mid = res[l] + atty Wproj^T + b.  At head size 64 (tensor-core
    // attention) its data gradient datty also yields the attention backward's
    // D = rowsum(datty * atty) per head, one head per 64-column group
    const bool fused_d = !f32 && C / NH == 64;
    GemmArgs gd = gemm(M, C, C, dres_act, C, true, w(ATTPROJW, (int64_t)l * C * C), C, false,
                       fused_d ? EPI_DOT_AUX : EPI_STORE, datty, C, f32);
    if (fused_d) {
      gd.aux = atty;
      gd.dot_out = m->dsum;
      gd.dot_T = T;
    }
    run_gemm(m, c, gd, GS_ATTPROJ);
    run_gemm(m, c, gemm(C, C, M, dres_act, C, false, atty, C, false, EPI_ACCUM,
                        m->G(ATTPROJW) + (int64_t)l * C * C, C, true), GS_ATTPROJ);
    // attproj bias gradient: taken by the LN2 backward above
    // attention (the tensor-core path also leaves the qkv bias gradient's
    // partial rows in its slot)
    bool qkvb_partials = false;
    float* qkvb_part = take_slot(std::max<int64_t>((int64_t)B * ((T + 127) / 128) * 3 * C, colsum_partial_floats(M, 3 * C)));
    {
      ProfScope ps(m, PC_ATTN_BWD, attn_flop);
      if (f32) launch_attention_bwd_simt<ActT>(c, dbig, datty, atty, qkv, lse, m->dsum, B, T, C, NH, nullptr);
      else qkvb_partials = launch_attention_bwd_bf16(c, reinterpret_cast<bf16*>(dbig), reinterpret_cast<const bf16*>(datty),
                                                     reinterpret_cast<const bf16*>(atty), reinterpret_cast<const bf16*>(qkv),
                                                     lse, m->dsum, fused_d, B, T, C, NH, qkvb_part);
    }
    // qkv: qkv = ln1 Wqkv^T + b
    run_gemm(m, c, gemm(M, C, 3 * C, dbig, 3 * C, true, w(QKVW, (int64_t)l * 3 * C * C), C, false,
                        EPI_STORE, dln, C, f32), GS_QKV);
    run_gemm(m, c, gemm(3 * C, C, M, dbig, 3 * C, false, ln1, C, false, EPI_ACCUM,
                        m->G(QKVW) + (int64_t)l * 3 * C * C, C, true), GS_QKV);
    if (qkvb_partials) {
      add_job(m->G(QKVB) + (int64_t)l * 3 * C, nullptr, nullptr, qkvb_part, B * ((T + 127) / 128), 3 * C, 3 * C);
    } else {
      ProfScope ps(m, PC_BIAS_GRAD, a * M * 3.0 * C);
      const int nb = launch_colsum_partials<ActT>(c, qkvb_part, dbig, M, 3 * C, 3 * C);
      add_job(m->G(QKVB) + (int64_t)l * 3 * C, nullptr, nullptr, qkvb_part, nb, 3 * C, 3 * C);
    }
    {
      ProfScope ps(m, PC_LN_BWD, lnb_bytes);
      float* part = take_slot(lnp);
      const int nb = launch_layernorm_bwd_partials<ActT>(c, m->dres, dres_act_out, dln, m->res[l], m->P(LN1W) + l * C,
                                                         m->ln1_mean + (int64_t)l * M, m->ln1_rstd + (int64_t)l * M,
                                                         M, C, true, part);
      add_job(m->G(LN1W) + l * C, m->G(LN1B) + l * C, l > 0 ? m->G(FCPROJB) + (int64_t)(l - 1) * C : nullptr, part,
              nb, 3 * C, C);
    }
  }
  {
    ProfScope ps(m, PC_ENC_BWD, 4.0 * M * C + 8.0 * T * C);
    launch_encoder_bwd(c, m->G(WTE), m->G(WPE), m->dres, m->tok, B, T, C, Vp, m->enc_sorted,
                       m->enc_partial);
  }
  {
    ProfScope ps(m, PC_BIAS_GRAD, 4.0 * (double)(slot - m->red_part));
    const int nj = (int)m->red_jobs.size();
    if (nj > m->red_jobs_cap) {
      c.host_fail = 1;
      return;
    }
    // the list is the same every pass: it goes to the device once
    if (m->red_jobs_up.size() != m->red_jobs.size() ||
        std::memcmp(m->red_jobs_up.data(), m->red_jobs.data(), sizeof(ReduceJob) * nj) != 0) {
      m->red_jobs_up = m->red_jobs;
      if (cudaMemcpyAsync(m->red_jobs_dev, m->red_jobs_up.data(), sizeof(ReduceJob) * nj, cudaMemcpyHostToDevice,
                          m->stream) != cudaSuccess)
        c.host_fail = 1;
    }
    launch_reduce_jobs(c, m->red_jobs_dev, nj, red_blocks);
  }
}

int forward_common(gpt2_model* m, bool with_targets, float* mean_loss) {
  LaunchCtx c = ctx(m);
  if (m->bf) forward_layers<bf16>(m, c, with_targets);
  else forward_layers<float>(m, c, with_targets);
  int rc = after_launches(m, c, "gpt2_forward");
  if (rc) return rc;
  m->have_fwd = true;
  m->have_cache = true;
  m->fwd_targets = with_targets;
  if (mean_loss) {
    rc = check_device(m, "gpt2_forward");
    if (rc) return rc;
    if (with_targets) {
      cudaError_t e = cudaMemcpy(mean_loss, m->loss, sizeof(float), cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_forward");
      if (!std::isfinite(*mean_loss)) return fail(m, GPT2_ERR_NONFINITE, "gpt2_forward: loss is not finite");
    } else {
      *mean_loss = NAN;
    }
  }
  return GPT2_OK;
}

}  // namespace

void set_global_error(const char* msg) { g_build_error = msg; }

// ====================================================================== ABI
extern "C" {

int gpt2_build(const gpt2_config* cfg, uint64_t seed, gpt2_model** out) {
  if (!out) return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: out is NULL");
  *out = nullptr;
  if (!cfg) return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: cfg is NULL");
  const gpt2_config& k = *cfg;
  const int hs = k.num_heads > 0 ? k.channels / k.num_heads : 0;
  if (k.num_layers < 1 || k.num_heads < 1 || k.channels < 8 || k.channels > 1024 ||
      k.channels % k.num_heads != 0 || k.channels % 8 != 0 ||
      !(hs == 16 || hs == 32 || hs == 64 || hs == 128))
    return fail(nullptr, GPT2_ERR_ARG,
                "gpt2_build: need L>=1, 8<=C<=1024, C%NH==0, C%8==0, head size in {16,32,64,128}");
  if (k.vocab_size < 1 || k.padded_vocab_size < k.vocab_size || k.padded_vocab_size % 8 != 0)
    return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: need 1 <= V <= Vp and Vp % 8 == 0");
  if (k.padded_vocab_size > (1 << 18))  // the encoder backward's radix sort takes 18-bit token ids
    return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: need Vp <= 262144");
  if (k.seq_len < 1 || k.seq_len > k.max_seq_len || k.max_seq_len > 4096 || k.batch_size < 1 ||
      (int64_t)k.batch_size * k.seq_len > 32768)
    return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: need 1 <= T <= maxT <= 4096, B >= 1, B*T <= 32768");
  if ((uint64_t)k.padded_vocab_size * (uint64_t)k.batch_size * (uint64_t)k.seq_len >= (1ull << 32))
    return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: Vp * B * T must be below 2^32");
  if (k.precision != GPT2_FP32 && k.precision != GPT2_BF16)
    return fail(nullptr, GPT2_ERR_ARG, "gpt2_build: unknown precision");
  if (k.precision == GPT2_BF16 && !gemm_bf16_init())
    return fail(nullptr, GPT2_ERR_CUDA, "gpt2_build: the driver's tensor-map encoder is unavailable");

  gpt2_model* m = new gpt2_model();
  m->cfg = k;
  m->L = k.num_layers; m->C = k.channels; m->NH = k.num_heads; m->V = k.vocab_size;
  m->Vp = k.padded_vocab_size; m->maxT = k.max_seq_len; m->B = k.batch_size; m->T = k.seq_len;
  m->M = m->B * m->T;
  m->bf = k.precision == GPT2_BF16;
  m->act = m->bf ? 2 : 4;
  cudaError_t e = cudaGetDevice(&m->device);
  if (e != cudaSuccess) { delete m; return cuda_fail(nullptr, e, "gpt2_build: cudaGetDevice"); }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, m->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, m->device);
  cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
  if (major != 10 || minor != 3) {
    delete m;
    return fail(nullptr, GPT2_ERR_CUDA, "gpt2_build: this library is built for sm_103 (B300) only");
  }
  int64_t n[NT];
  param_sizes(m, n);
  m->off[0] = 0;
  for (int t = 0; t < NT; t++) m->off[t + 1] = m->off[t] + n[t];
  m->n_params = m->off[NT];
  m->block_bytes = layout(m, nullptr);
  e = cudaMalloc(&m->block, m->block_bytes);
  if (e != cudaSuccess) {
    delete m;
    cudaGetLastError();
    return fail(nullptr, GPT2_ERR_OOM, "gpt2_build: cudaMalloc of the model block failed");
  }
  layout(m, m->block);
  cudaMemset(m->grads, 0, sizeof(float) * m->n_params);
  cudaMemset(m->adam_m, 0, sizeof(float) * m->n_params);
  cudaMemset(m->adam_v, 0, sizeof(float) * m->n_params);
  cudaMemset(m->err, 0, sizeof(int));
  if (m->splitk_flag_count) cudaMemset(m->splitk_flags, 0, sizeof(int) * m->splitk_flag_count);
  LaunchCtx c = ctx(m);
  InitSpec s;
  for (int t = 0; t <= NT; t++) s.off[t] = m->off[t];
  s.L = m->L; s.C = m->C; s.V = m->V; s.seed = seed;
  launch_init_params(c, m->params, s);
  if (m->bf) launch_f32_to_bf16(c, m->wb, m->params, m->n_params);
  int rc = after_launches(m, c, "gpt2_build");
  if (rc == GPT2_OK) rc = check_device(m, "gpt2_build");
  if (rc != GPT2_OK) {
    g_build_error = m->last_error;
    cudaFree(m->block);
    delete m;
    return rc;
  }
  *out = m;
  return GPT2_OK;
}

void gpt2_free(gpt2_model* m) {
  if (!m) return;
  cudaSetDevice(m->device);
  cudaStreamSynchronize(m->stream);
  for (auto& p : m->prof.pending) { cudaEventDestroy(p.second.first); cudaEventDestroy(p.second.second); }
  for (cudaEvent_t e : m->prof.pool) cudaEventDestroy(e);
  if (m->dec_exec) cudaGraphExecDestroy(m->dec_exec);
  if (m->dec_graph) cudaGraphDestroy(m->dec_graph);
  if (m->dec_cap) cudaStreamDestroy(m->dec_cap);
  cudaFree(m->block);
  delete m;
}

int gpt2_set_stream(gpt2_model* m, void* s) {
  if (!m) return GPT2_ERR_ARG;
  m->stream = static_cast<cudaStream_t>(s);
  return GPT2_OK;
}

int gpt2_forward(gpt2_model* m, const int32_t* tokens, const int32_t* targets, float* mean_loss) {
  if (!m) return GPT2_ERR_ARG;
  if (!tokens) return fail(m, GPT2_ERR_ARG, "gpt2_forward: tokens is NULL");
  cudaSetDevice(m->device);
  cudaError_t e = cudaMemcpyAsync(m->tok, tokens, sizeof(int32_t) * m->M, cudaMemcpyDeviceToDevice, m->stream);
  if (e == cudaSuccess && targets)
    e = cudaMemcpyAsync(m->tgt, targets, sizeof(int32_t) * m->M, cudaMemcpyDeviceToDevice, m->stream);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_forward: copying ids");
  return forward_common(m, targets != nullptr, mean_loss);
}

int gpt2_forward_host(gpt2_model* m, const int32_t* tokens, const int32_t* targets, float* mean_loss) {
  if (!m) return GPT2_ERR_ARG;
  if (!tokens) return fail(m, GPT2_ERR_ARG, "gpt2_forward_host: tokens is NULL");
  cudaSetDevice(m->device);
  cudaError_t e = cudaMemcpyAsync(m->tok, tokens, sizeof(int32_t) * m->M, cudaMemcpyHostToDevice, m->stream);
  if (e == cudaSuccess && targets)
    e = cudaMemcpyAsync(m->tgt, targets, sizeof(int32_t) * m->M, cudaMemcpyHostToDevice, m->stream);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_forward_host: copying ids");
  return forward_common(m, targets != nullptr, mean_loss);
}

int gpt2_zero_grad(gpt2_model* m) {
  if (!m) return GPT2_ERR_ARG;
  cudaSetDevice(m->device);
  cudaError_t e;
  {
    ProfScope ps(m, PC_ZERO_GRAD, 4.0 * m->n_params);
    e = cudaMemsetAsync(m->grads, 0, sizeof(float) * m->n_params, m->stream);
  }
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_zero_grad");
  return GPT2_OK;
}

int gpt2_backward(gpt2_model* m) {
  if (!m) return GPT2_ERR_ARG;
  if (!m->have_fwd || !m->fwd_targets)
    return fail(m, GPT2_ERR_STATE, "gpt2_backward: needs a preceding forward with targets");
  cudaSetDevice(m->device);
  LaunchCtx c = ctx(m);
  if (m->bf) backward_layers<bf16>(m, c);
  else backward_layers<float>(m, c);
  m->have_fwd = false;  // the dlogits buffer has been consumed
  return after_launches(m, c, "gpt2_backward");
}

int gpt2_adamw_step(gpt2_model* m, float lr, float b1, float b2, float eps, float wd, int32_t t) {
  if (!m) return GPT2_ERR_ARG;
  if (t < 1) return fail(m, GPT2_ERR_ARG, "gpt2_adamw_step: t must be >= 1");
  if (!std::isfinite(lr) || !std::isfinite(b1) || !std::isfinite(b2) || !std::isfinite(eps) ||
      !std::isfinite(wd))
    return fail(m, GPT2_ERR_ARG, "gpt2_adamw_step: non-finite hyper-parameter");
  cudaSetDevice(m->device);
  LaunchCtx c = ctx(m);
  const float c1 = 1.f - powf(b1, (float)t), c2 = 1.f - powf(b2, (float)t);
  {
    ProfScope ps(m, PC_ADAMW, (28.0 + (m->bf ? 2.0 : 0.0)) * m->n_params);
    launch_adamw(c, m->params, m->grads, m->adam_m, m->adam_v, m->bf ? m->wb : nullptr, m->n_params,
                 lr, b1, b2, eps, wd, c1, c2);
  }
  m->have_cache = false;  // keys / values of the old weights
  return after_launches(m, c, "gpt2_adamw_step");
}

int gpt2_synchronize(gpt2_model* m) {
  if (!m) return GPT2_ERR_ARG;
  cudaSetDevice(m->device);
  return check_device(m, "gpt2_synchronize");
}

int gpt2_expire_a_wait(gpt2_model* m) {
  if (!m) return GPT2_ERR_ARG;
  cudaSetDevice(m->device);
  LaunchCtx c = ctx(m);
  launch_expire_wait(c);
  return after_launches(m, c, "gpt2_expire_a_wait");
}

int gpt2_get_config(const gpt2_model* m, gpt2_config* out) {
  if (!m || !out) return GPT2_ERR_ARG;
  *out = m->cfg;
  return GPT2_OK;
}

int gpt2_num_params(const gpt2_model* m, int64_t* n) {
  if (!m || !n) return GPT2_ERR_ARG;
  *n = m->n_params;
  return GPT2_OK;
}

int gpt2_num_tensors(const gpt2_model* m, int32_t* n) {
  if (!m || !n) return GPT2_ERR_ARG;
  *n = NT;
  return GPT2_OK;
}

int gpt2_tensor_info(const gpt2_model* m, int32_t idx, const char** name, int64_t* offset,
                     int64_t* numel) {
  if (!m || idx < 0 || idx >= NT) return GPT2_ERR_ARG;
  if (name) *name = kTensorNames[idx];
  if (offset) *offset = m->off[idx];
  if (numel) *numel = m->off[idx + 1] - m->off[idx];
  return GPT2_OK;
}

static float* arena_ptr(gpt2_model* m, int32_t a) {
  switch (a) {
    case GPT2_PARAMS: return m->params;
    case GPT2_GRADS: return m->grads;
    case GPT2_ADAM_M: return m->adam_m;
    case GPT2_ADAM_V: return m->adam_v;
  }
  return nullptr;
}

int gpt2_copy_out(gpt2_model* m, int32_t arena, float* dst) {
  if (!m) return GPT2_ERR_ARG;
  float* src = arena_ptr(m, arena);
  if (!src || !dst) return fail(m, GPT2_ERR_ARG, "gpt2_copy_out: bad arena or NULL destination");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_copy_out");
  if (rc) return rc;
  cudaError_t e = cudaMemcpy(dst, src, sizeof(float) * m->n_params, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? GPT2_OK : cuda_fail(m, e, "gpt2_copy_out");
}

int gpt2_copy_in(gpt2_model* m, int32_t arena, const float* srch) {
  if (!m) return GPT2_ERR_ARG;
  float* dst = arena_ptr(m, arena);
  if (!dst || !srch) return fail(m, GPT2_ERR_ARG, "gpt2_copy_in: bad arena or NULL source");
  cudaSetDevice(m->device);
  cudaError_t e = cudaStreamSynchronize(m->stream);
  if (e == cudaSuccess) e = cudaMemcpy(dst, srch, sizeof(float) * m->n_params, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_copy_in");
  if (arena == GPT2_PARAMS) m->have_cache = false;
  if (arena == GPT2_PARAMS && m->bf) {
    LaunchCtx c = ctx(m);
    launch_f32_to_bf16(c, m->wb, m->params, m->n_params);
    int rc = after_launches(m, c, "gpt2_copy_in");
    if (rc) return rc;
  }
  return check_device(m, "gpt2_copy_in");
}

// ---------------------------------------------------------------- checkpoints
// Header and arena layout: see gpt2_save_checkpoint in gpt2.h.
#define CKPT_MAGIC 0x43545047  // "GPTC"
#define CKPT_VERSION 1
#define CKPT_HEADER 64
#define CKPT_CHUNK (1 << 24)  // floats per host staging chunk (64 MB)

static void ckpt_header(const gpt2_model* m, int32_t step, int32_t* h) {
  std::memset(h, 0, sizeof(int32_t) * CKPT_HEADER);
  const gpt2_config& k = m->cfg;
  h[0] = CKPT_MAGIC; h[1] = CKPT_VERSION; h[2] = CKPT_HEADER;
  h[3] = k.max_seq_len; h[4] = k.vocab_size; h[5] = k.padded_vocab_size; h[6] = k.num_layers;
  h[7] = k.num_heads; h[8] = k.channels; h[9] = k.batch_size; h[10] = k.seq_len; h[11] = k.precision;
  h[12] = step;
  h[13] = (int32_t)(uint32_t)((uint64_t)m->n_params & 0xffffffffu);
  h[14] = (int32_t)(uint32_t)((uint64_t)m->n_params >> 32);
  h[15] = 3;
}

int gpt2_save_checkpoint(gpt2_model* m, const char* path, int32_t step) {
  if (!m) return GPT2_ERR_ARG;
  if (!path || step < 0) return fail(m, GPT2_ERR_ARG, "gpt2_save_checkpoint: NULL path or step < 0");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_save_checkpoint");
  if (rc) return rc;
  FILE* f = std::fopen(path, "wb");
  if (!f) return fail(m, GPT2_ERR_IO, std::string("gpt2_save_checkpoint: cannot open ") + path);
  int32_t h[CKPT_HEADER];
  ckpt_header(m, step, h);
  bool ok = std::fwrite(h, sizeof(int32_t), CKPT_HEADER, f) == CKPT_HEADER;
  std::vector<float> buf((size_t)std::min<int64_t>(m->n_params, CKPT_CHUNK));
  const float* arenas[3] = {m->params, m->adam_m, m->adam_v};
  cudaError_t e = cudaSuccess;
  for (int a = 0; a < 3 && ok && e == cudaSuccess; a++) {
    for (int64_t i = 0; i < m->n_params && ok; i += CKPT_CHUNK) {
      const size_t n = (size_t)std::min<int64_t>(CKPT_CHUNK, m->n_params - i);
      e = cudaMemcpy(buf.data(), arenas[a] + i, n * sizeof(float), cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) break;
      ok = std::fwrite(buf.data(), sizeof(float), n, f) == n;
    }
  }
  ok = (std::fclose(f) == 0) && ok;
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_save_checkpoint");
  if (!ok) return fail(m, GPT2_ERR_IO, std::string("gpt2_save_checkpoint: write failed: ") + path);
  return GPT2_OK;
}

int gpt2_load_checkpoint(gpt2_model* m, const char* path, int32_t* step) {
  if (!m) return GPT2_ERR_ARG;
  if (!path) return fail(m, GPT2_ERR_ARG, "gpt2_load_checkpoint: NULL path");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_load_checkpoint");
  if (rc) return rc;
  FILE* f = std::fopen(path, "rb");
  if (!f) return fail(m, GPT2_ERR_IO, std::string("gpt2_load_checkpoint: cannot open ") + path);
  int32_t h[CKPT_HEADER], want[CKPT_HEADER];
  if (std::fread(h, sizeof(int32_t), CKPT_HEADER, f) != CKPT_HEADER) {
    std::fclose(f);
    return fail(m, GPT2_ERR_IO, "gpt2_load_checkpoint: short header");
  }
  ckpt_header(m, h[12], want);
  bool match = h[0] == want[0] && h[1] == want[1] && h[2] == want[2] && h[15] == want[15] && h[12] >= 0;
  for (int i = 3; i <= 8; i++) match = match && h[i] == want[i];  // model shape
  match = match && h[13] == want[13] && h[14] == want[14];        // parameter count
  if (!match) {
    std::fclose(f);
    return fail(m, GPT2_ERR_ARG, "gpt2_load_checkpoint: not a checkpoint of this model's shape");
  }
  // the whole file is there before anything of the model is replaced
  std::fseek(f, 0, SEEK_END);
  const long long bytes = (long long)std::ftell(f);
  std::fseek(f, (long)(sizeof(int32_t) * CKPT_HEADER), SEEK_SET);
  if (bytes < (long long)(sizeof(int32_t) * CKPT_HEADER) + 3LL * (long long)sizeof(float) * m->n_params) {
    std::fclose(f);
    return fail(m, GPT2_ERR_IO, "gpt2_load_checkpoint: file ends before the arenas do");
  }
  std::vector<float> buf((size_t)std::min<int64_t>(m->n_params, CKPT_CHUNK));
  float* arenas[3] = {m->params, m->adam_m, m->adam_v};
  bool ok = true;
  cudaError_t e = cudaSuccess;
  for (int a = 0; a < 3 && ok && e == cudaSuccess; a++) {
    for (int64_t i = 0; i < m->n_params && ok; i += CKPT_CHUNK) {
      const size_t n = (size_t)std::min<int64_t>(CKPT_CHUNK, m->n_params - i);
      ok = std::fread(buf.data(), sizeof(float), n, f) == n;
      if (ok) e = cudaMemcpy(arenas[a] + i, buf.data(), n * sizeof(float), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) break;
    }
  }
  std::fclose(f);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_load_checkpoint");
  if (!ok) return fail(m, GPT2_ERR_IO, "gpt2_load_checkpoint: file ends before the arenas do");
  e = cudaMemsetAsync(m->grads, 0, sizeof(float) * m->n_params, m->stream);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_load_checkpoint");
  if (m->bf) {
    LaunchCtx c = ctx(m);
    launch_f32_to_bf16(c, m->wb, m->params, m->n_params);
    rc = after_launches(m, c, "gpt2_load_checkpoint");
    if (rc) return rc;
  }
  m->have_fwd = false;
  m->have_cache = false;
  rc = check_device(m, "gpt2_load_checkpoint");
  if (rc) return rc;
  if (step) *step = h[12];
  return GPT2_OK;
}

// Record the decode step's launches once into a CUDA graph (on a private
// stream); they read the step's inputs from the model's buffers.
static int capture_decode(gpt2_model* m) {
  cudaError_t e = cudaSuccess;
  if (!m->dec_cap) e = cudaStreamCreateWithFlags(&m->dec_cap, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_decode_step: stream");
  LaunchCtx c = ctx(m);
  c.stream = m->dec_cap;
  const int64_t l0 = m->launches;
  e = cudaStreamBeginCapture(m->dec_cap, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_decode_step: begin capture");
  if (m->bf) decode_layers<bf16>(m, c, true, 0);
  else decode_layers<float>(m, c, true, 0);
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(m->dec_cap, &graph);
  const int64_t n = m->launches - l0;
  m->launches = l0;  // counted when the graph is launched
  if (e != cudaSuccess || c.host_fail || !graph) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return fail(m, GPT2_ERR_CUDA, "gpt2_decode_step: capturing the step failed");
  }
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_fail(m, e, "gpt2_decode_step: graph instantiation");
  }
  m->dec_graph = graph;
  m->dec_exec = exec;
  m->dec_graph_launches = n;
  return GPT2_OK;
}

int gpt2_decode_step(gpt2_model* m, const int32_t* tokens, int32_t pos, float temperature,
                     const float* uniforms, int32_t* next_tokens) {
  if (!m) return GPT2_ERR_ARG;
  if (!tokens || !uniforms || !next_tokens) return fail(m, GPT2_ERR_ARG, "gpt2_decode_step: NULL pointer");
  if (pos < 0 || pos >= m->T) return fail(m, GPT2_ERR_ARG, "gpt2_decode_step: pos outside [0, T)");
  if (!std::isfinite(temperature)) return fail(m, GPT2_ERR_ARG, "gpt2_decode_step: temperature is not finite");
  if (!m->have_cache)
    return fail(m, GPT2_ERR_STATE, "gpt2_decode_step: no key/value cache of the current weights (run gpt2_forward first)");
  cudaSetDevice(m->device);
  LaunchCtx c = ctx(m);
  launch_decode_inputs(c, m->dec_tok, tokens, m->dec_u, uniforms, m->dec_pos, pos, m->dec_temp, temperature, m->B);
  int rc = after_launches(m, c, "gpt2_decode_step");
  if (rc) return rc;
  // replayed as one graph unless kernel classes are being timed (events per
  // launch) or the few-row matmul does not apply (more than 16 sequences)
  const bool graph = m->prof.mask == 0 && (!m->bf || m->B <= 16);
  if (graph) {
    if (!m->dec_exec) {
      rc = capture_decode(m);
      if (rc) return rc;
    }
    cudaError_t e = cudaGraphLaunch(m->dec_exec, m->stream);
    if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_decode_step: graph launch");
    m->launches += m->dec_graph_launches;
  } else {
    if (m->bf) decode_layers<bf16>(m, c, false, pos);
    else decode_layers<float>(m, c, false, pos);
    rc = after_launches(m, c, "gpt2_decode_step");
    if (rc) return rc;
  }
  cudaError_t e = cudaMemcpyAsync(next_tokens, m->dec_next, sizeof(int32_t) * m->B, cudaMemcpyDeviceToDevice, m->stream);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_decode_step: copying the drawn ids");
  // row pos of the cache now holds the new position: the activations of the
  // last forward no longer match each other
  m->have_fwd = false;
  m->fwd_targets = false;
  m->have_dec = true;
  return GPT2_OK;
}

int gpt2_copy_decode_logits_out(gpt2_model* m, float* dst) {
  if (!m || !dst) return GPT2_ERR_ARG;
  if (!m->have_dec) return fail(m, GPT2_ERR_STATE, "gpt2_copy_decode_logits_out: no decode step to read");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_copy_decode_logits_out");
  if (rc) return rc;
  const size_t n = (size_t)m->B * m->Vp;
  if (!m->bf) {
    cudaError_t e = cudaMemcpy(dst, m->dec_logits, sizeof(float) * n, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? GPT2_OK : cuda_fail(m, e, "gpt2_copy_decode_logits_out");
  }
  std::vector<uint16_t> tmp(n);
  cudaError_t e = cudaMemcpy(tmp.data(), m->dec_logits, 2 * n, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_copy_decode_logits_out");
  for (size_t i = 0; i < n; i++) {
    uint32_t u = (uint32_t)tmp[i] << 16;
    std::memcpy(&dst[i], &u, 4);
  }
  return GPT2_OK;
}

int gpt2_copy_losses_out(gpt2_model* m, float* dst) {
  if (!m || !dst) return GPT2_ERR_ARG;
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_copy_losses_out");
  if (rc) return rc;
  cudaError_t e = cudaMemcpy(dst, m->losses, sizeof(float) * m->M, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? GPT2_OK : cuda_fail(m, e, "gpt2_copy_losses_out");
}

int gpt2_copy_logits_out(gpt2_model* m, float* dst) {
  if (!m || !dst) return GPT2_ERR_ARG;
  if (!m->have_fwd || m->fwd_targets)
    return fail(m, GPT2_ERR_STATE, "gpt2_copy_logits_out: needs a preceding forward without targets");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_copy_logits_out");
  if (rc) return rc;
  const size_t n = (size_t)m->M * m->Vp;
  if (!m->bf) {
    cudaError_t e = cudaMemcpy(dst, m->logits, sizeof(float) * n, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? GPT2_OK : cuda_fail(m, e, "gpt2_copy_logits_out");
  }
  std::vector<uint16_t> tmp(n);
  cudaError_t e = cudaMemcpy(tmp.data(), m->logits, 2 * n, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_copy_logits_out");
  for (size_t i = 0; i < n; i++) {
    uint32_t u = (uint32_t)tmp[i] << 16;
    std::memcpy(&dst[i], &u, 4);
  }
  return GPT2_OK;
}

int gpt2_copy_residual_out(gpt2_model* m, int32_t layer, float* dst) {
  if (!m || !dst) return GPT2_ERR_ARG;
  if (layer < 0 || layer > m->L) return fail(m, GPT2_ERR_ARG, "gpt2_copy_residual_out: layer outside [0, L]");
  if (!m->have_fwd) return fail(m, GPT2_ERR_STATE, "gpt2_copy_residual_out: no forward to read");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_copy_residual_out");
  if (rc) return rc;
  cudaError_t e = cudaMemcpy(dst, m->res[layer], sizeof(float) * (size_t)m->M * m->C, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? GPT2_OK : cuda_fail(m, e, "gpt2_copy_residual_out");
}

int gpt2_copy_params_out(gpt2_model* m, float* dst) { return gpt2_copy_out(m, GPT2_PARAMS, dst); }
int gpt2_copy_grads_out(gpt2_model* m, float* dst) { return gpt2_copy_out(m, GPT2_GRADS, dst); }
int gpt2_copy_m_out(gpt2_model* m, float* dst) { return gpt2_copy_out(m, GPT2_ADAM_M, dst); }
int gpt2_copy_v_out(gpt2_model* m, float* dst) { return gpt2_copy_out(m, GPT2_ADAM_V, dst); }
int gpt2_copy_params_in(gpt2_model* m, const float* src) { return gpt2_copy_in(m, GPT2_PARAMS, src); }

int gpt2_loss_device_ptr(const gpt2_model* m, const float** out) {
  if (!m || !out) return GPT2_ERR_ARG;
  *out = m->loss;
  return GPT2_OK;
}

int gpt2_read_loss(gpt2_model* m, float* host_loss) {
  if (!m || !host_loss) return GPT2_ERR_ARG;
  if (!m->fwd_targets) return fail(m, GPT2_ERR_STATE, "gpt2_read_loss: no forward with targets");
  cudaSetDevice(m->device);
  int rc = check_device(m, "gpt2_read_loss");
  if (rc) return rc;
  cudaError_t e = cudaMemcpy(host_loss, m->loss, sizeof(float), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_read_loss");
  if (!std::isfinite(*host_loss)) return fail(m, GPT2_ERR_NONFINITE, "gpt2_read_loss: loss is not finite");
  return GPT2_OK;
}

int gpt2_profile_num_classes(int32_t* n) {
  if (!n) return GPT2_ERR_ARG;
  *n = PC_N;
  return GPT2_OK;
}

int gpt2_profile_enable(gpt2_model* m, uint32_t mask) {
  if (!m) return GPT2_ERR_ARG;
  m->prof.mask = mask & ((1u << PC_N) - 1u);
  return GPT2_OK;
}

static int profile_collect(gpt2_model* m) {
  cudaError_t e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) return cuda_fail(m, e, "gpt2_profile_read");
  for (auto& p : m->prof.pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.second.first, p.second.second) == cudaSuccess) m->prof.ms[p.first] += ms;
    m->prof.pool.push_back(p.second.first);
    m->prof.pool.push_back(p.second.second);
  }
  m->prof.pending.clear();
  return GPT2_OK;
}

int gpt2_profile_reset(gpt2_model* m) {
  if (!m) return GPT2_ERR_ARG;
  cudaSetDevice(m->device);
  int rc = profile_collect(m);
  for (int i = 0; i < PC_N; i++) { m->prof.launches[i] = 0; m->prof.work[i] = 0; m->prof.ms[i] = 0; }
  return rc;
}

int gpt2_profile_read(gpt2_model* m, int32_t cls, const char** name, const char** unit,
                      int64_t* launches, double* total_ms, double* work) {
  if (!m || cls < 0 || cls >= PC_N) return GPT2_ERR_ARG;
  cudaSetDevice(m->device);
  int rc = profile_collect(m);
  if (rc) return rc;
  if (name) *name = kProfNames[cls];
  if (unit) *unit = kProfUnits[cls];
  if (launches) *launches = m->prof.launches[cls];
  if (total_ms) *total_ms = m->prof.ms[cls];
  if (work) *work = m->prof.work[cls];
  return GPT2_OK;
}

int gpt2_launch_count(const gpt2_model* m, int64_t* n) {
  if (!m || !n) return GPT2_ERR_ARG;
  *n = m->launches;
  return GPT2_OK;
}

const char* gpt2_last_error(const gpt2_model* m) {
  return m ? m->last_error.c_str() : g_build_error.c_str();
}

}  // extern "C"
