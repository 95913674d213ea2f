/*
 * gpt2_oracle.cpp -- the ORACLE for one GPT-2 training step.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path (the
 * CUDA library under transformer_lm_step_gpt_b300/csrc) never links, includes
 * or calls anything here, and nothing here includes or calls the product.
 *
 * What it is: a plain, slow, obviously-correct CPU implementation of the
 * method, templated over float (the fp32 oracle) and double (used for the
 * finite-difference and library cross-checks).  Every reduction is a plain
 * sequential loop in the element order of its formula; OpenMP only splits
 * loops over *independent outputs*, so results do not depend on the thread
 * count.  No blocking, fusion or reordering beyond what the formulas state.
 *
 * Sources (the pages this restates; cited by title and section):
 *  [QbitAI]   QbitAI, "OpenAI founder hand-writes a thousand lines of C to
 *             train GPT, with a PyTorch migration tutorial" (2024-04-09),
 *             section "Manually implementing each layer's forward/backward
 *             pass": one 1-D allocation holds every weight and activation;
 *             each layer has a hand-written forward and backward, chained.
 *  [InfoQ]    InfoQ, "Real men program in C: a large model hand-built from
 *             1000 lines of C", the paragraph naming the layers (layernorm,
 *             encoder, matmul, self-attention, gelu, residual, softmax,
 *             cross-entropy loss), the fine-tuning loop ("Adam lr 1e-4") and
 *             the M3 Max run log (num_parameters, num_activations).
 *  [GeekNews] GeekNews, "A GPT-2-based ChatGPT clone in 3000 bytes of C
 *             (2023)", sections "Implementing the neural-network layers"
 *             (GELU, lower-triangular causal mask, LayerNorm, Linear adds a
 *             bias tiled over rows), "The Transformer core" (block order,
 *             final LayerNorm, product with the embedding matrix) and the
 *             Hacker News comments (the tanh form of GELU, GELU = x*Phi(x)).
 *  [microgpt] "microgpt" (aiviet.app), introduction: an Adam optimiser.
 *  [femtoGPT] "femtoGPT: a minimal generative pretrained Transformer in pure
 *             Rust", section "Gradient checking" (the test method used to
 *             pin the backward passes, see tests/test_oracle_grad.py).
 *
 * Readings where the pages are silent:
 *  - pre-LN block: x += proj(attn(LN1(x))); x += fcproj(GELU(fc(LN2(x))));
 *    then LN_f and the tied head logits = LN_f(x) * wte^T (no head bias);
 *  - LayerNorm: biased variance (divide by C), eps = 1e-5 inside the sqrt;
 *  - GELU: the tanh form with sqrt(2/pi) at full precision and 0.044715;
 *  - attention scale 1/sqrt(hs); position i attends to j <= i;
 *  - Linear: y = x W^T + b with W row-major [out, in];
 *  - the loss is the mean over all B*T positions; pad vocabulary columns
 *    (V <= j < Vp) are not part of the softmax;
 *  - AdamW: m, v moments, bias correction with 1-based t, eps outside the
 *    sqrt, decoupled weight decay on every parameter using the pre-update p.
 *
 * This file is pinned against the mathematics and the pages' printed numbers
 * by the tests marked "not gpu" (tests/test_oracle_*.py).
 */
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------- shapes

struct Shape {
  int64_t L, C, NH, V, Vp, maxT, B, T;
};

// cfg8 = {L, C, NH, V, Vp, maxT, B, T}
Shape shape_from(const int32_t* cfg8) {
  Shape s;
  s.L = cfg8[0]; s.C = cfg8[1]; s.NH = cfg8[2]; s.V = cfg8[3];
  s.Vp = cfg8[4]; s.maxT = cfg8[5]; s.B = cfg8[6]; s.T = cfg8[7];
  return s;
}

bool shape_ok(const Shape& s) {
  return s.L >= 0 && s.C > 0 && s.NH > 0 && s.C % s.NH == 0 && s.V > 0 &&
         s.Vp >= s.V && s.maxT > 0 && s.B > 0 && s.T > 0 && s.T <= s.maxT;
}

// The parameter tensors, in the order they sit in the single 1-D parameter
// array ([QbitAI]: one allocation, every weight a pointer into it).  The set
// of tensors is the one whose size reproduces the printed num_parameters of
// the [InfoQ] run log: tied embedding (no separate head), biases on all four
// Linears, gamma/beta on both block LayerNorms and on the final one, learned
// position embedding.
enum ParamId {
  WTE = 0, WPE, LN1W, LN1B, QKVW, QKVB, ATTPROJW, ATTPROJB,
  LN2W, LN2B, FCW, FCB, FCPROJW, FCPROJB, LNFW, LNFB, NUM_PARAMS
};

void param_sizes(const Shape& s, int64_t n[NUM_PARAMS]) {
  const int64_t L = s.L, C = s.C;
  n[WTE] = s.Vp * C;      n[WPE] = s.maxT * C;
  n[LN1W] = L * C;        n[LN1B] = L * C;
  n[QKVW] = L * 3 * C * C; n[QKVB] = L * 3 * C;
  n[ATTPROJW] = L * C * C; n[ATTPROJB] = L * C;
  n[LN2W] = L * C;        n[LN2B] = L * C;
  n[FCW] = L * 4 * C * C; n[FCB] = L * 4 * C;
  n[FCPROJW] = L * C * 4 * C; n[FCPROJB] = L * C;
  n[LNFW] = C;            n[LNFB] = C;
}

// The plain, fully materialised activation set (every intermediate of the
// forward pass kept for the backward pass), as one more 1-D array.  Its size
// at the [InfoQ] run-log shape is the printed num_activations.
enum ActId {
  ENCODED = 0, LN1, LN1_MEAN, LN1_RSTD, QKV, ATTY, PREATT, ATT, ATTPROJ,
  RESIDUAL2, LN2, LN2_MEAN, LN2_RSTD, FCH, FCH_GELU, FCPROJ, RESIDUAL3,
  LNF, LNF_MEAN, LNF_RSTD, LOGITS, PROBS, LOSSES, NUM_ACTS
};

void act_sizes(const Shape& s, int64_t n[NUM_ACTS]) {
  const int64_t L = s.L, C = s.C, BT = s.B * s.T, NH = s.NH, T = s.T;
  n[ENCODED] = BT * C;
  n[LN1] = L * BT * C;  n[LN1_MEAN] = L * BT;  n[LN1_RSTD] = L * BT;
  n[QKV] = L * BT * 3 * C;
  n[ATTY] = L * BT * C;
  n[PREATT] = L * s.B * NH * T * T;  n[ATT] = L * s.B * NH * T * T;
  n[ATTPROJ] = L * BT * C;  n[RESIDUAL2] = L * BT * C;
  n[LN2] = L * BT * C;  n[LN2_MEAN] = L * BT;  n[LN2_RSTD] = L * BT;
  n[FCH] = L * BT * 4 * C;  n[FCH_GELU] = L * BT * 4 * C;
  n[FCPROJ] = L * BT * C;  n[RESIDUAL3] = L * BT * C;
  n[LNF] = BT * C;  n[LNF_MEAN] = BT;  n[LNF_RSTD] = BT;
  n[LOGITS] = BT * s.V;  n[PROBS] = BT * s.V;  n[LOSSES] = BT;
}

template <typename R>
struct Tensors {
  std::vector<R*> p;
  Tensors(R* base, const int64_t* sizes, int count) : p(count) {
    R* q = base;
    for (int i = 0; i < count; i++) { p[i] = q; q += sizes[i]; }
  }
  R* operator[](int i) const { return p[i]; }
};

const double kLnEps = 1e-5;

// ---------------------------------------------------------------- layers

// encoder: token embedding plus position embedding ([InfoQ] layer list).
template <typename R>
void encoder_forward(R* out, const int32_t* tok, const R* wte, const R* wpe,
                     int64_t B, int64_t T, int64_t C) {
  for (int64_t b = 0; b < B; b++)
    for (int64_t t = 0; t < T; t++) {
      const R* e = wte + (int64_t)tok[b * T + t] * C;
      const R* p = wpe + t * C;
      R* o = out + (b * T + t) * C;
      for (int64_t c = 0; c < C; c++) o[c] = e[c] + p[c];
    }
}

// The gradient of a sum of looked-up rows: every position adds its
// gradient row into the row of its token and into the row of its position.
template <typename R>
void encoder_backward(R* dwte, R* dwpe, const R* dout, const int32_t* tok,
                      int64_t B, int64_t T, int64_t C) {
  for (int64_t b = 0; b < B; b++)
    for (int64_t t = 0; t < T; t++) {
      const R* d = dout + (b * T + t) * C;
      R* dw = dwte + (int64_t)tok[b * T + t] * C;
      R* dp = dwpe + t * C;
      for (int64_t c = 0; c < C; c++) { dw[c] += d[c]; dp[c] += d[c]; }
    }
}

// LayerNorm ([QbitAI] worked example; [GeekNews] "normalises the mean and
// variance"): mu = mean(x), var = mean((x-mu)^2), r = 1/sqrt(var+eps),
// y = (x-mu)*r*gamma + beta.  Two passes over the row.
template <typename R>
void layernorm_forward(R* out, R* mean, R* rstd, const R* inp, const R* w,
                       const R* b, int64_t N, int64_t C) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; i++) {
    const R* x = inp + i * C;
    R m = 0;
    for (int64_t c = 0; c < C; c++) m += x[c];
    m = m / (R)C;
    R v = 0;
    for (int64_t c = 0; c < C; c++) { R d = x[c] - m; v += d * d; }
    v = v / (R)C;
    R r = (R)1 / std::sqrt(v + (R)kLnEps);
    R* y = out + i * C;
    for (int64_t c = 0; c < C; c++) y[c] = (x[c] - m) * r * w[c] + b[c];
    mean[i] = m;
    rstd[i] = r;
  }
}

// LayerNorm backward.  With xhat = (x-mu)*r and g = dy*gamma:
//   dx     += r * (g - mean(g) - xhat * mean(g*xhat))
//   dgamma += sum_rows dy * xhat,   dbeta += sum_rows dy.
template <typename R>
void layernorm_backward(R* dinp, R* dw, R* db, const R* dout, const R* inp,
                        const R* w, const R* mean, const R* rstd, int64_t N,
                        int64_t C) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; i++) {
    const R* x = inp + i * C;
    const R* dy = dout + i * C;
    const R m = mean[i], r = rstd[i];
    R mg = 0, mgx = 0;
    for (int64_t c = 0; c < C; c++) {
      R xhat = (x[c] - m) * r;
      R g = dy[c] * w[c];
      mg += g;
      mgx += g * xhat;
    }
    mg = mg / (R)C;
    mgx = mgx / (R)C;
    R* dx = dinp + i * C;
    for (int64_t c = 0; c < C; c++) {
      R xhat = (x[c] - m) * r;
      R g = dy[c] * w[c];
      dx[c] += r * (g - mg - xhat * mgx);
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < C; c++) {
    R sw = 0, sb = 0;
    for (int64_t i = 0; i < N; i++) {
      R xhat = (inp[i * C + c] - mean[i]) * rstd[i];
      sw += dout[i * C + c] * xhat;
      sb += dout[i * C + c];
    }
    dw[c] += sw;
    db[c] += sb;
  }
}

// Linear ([GeekNews]: a matrix product, then a bias tiled over the rows):
//   out[n, o] = sum_i inp[n, i] * W[o, i] + bias[o].   bias may be null.
template <typename R>
void matmul_forward(R* out, const R* inp, const R* W, const R* bias,
                    int64_t N, int64_t IC, int64_t OC) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; n++) {
    const R* x = inp + n * IC;
    for (int64_t o = 0; o < OC; o++) {
      const R* wr = W + o * IC;
      R s = 0;
      for (int64_t i = 0; i < IC; i++) s += x[i] * wr[i];
      out[n * OC + o] = bias ? s + bias[o] : s;
    }
  }
}

// Linear backward: dinp += dout W;  dW += dout^T inp;  dbias += sum_n dout.
template <typename R>
void matmul_backward(R* dinp, R* dW, R* dbias, const R* dout, const R* inp,
                     const R* W, int64_t N, int64_t IC, int64_t OC) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; n++) {
    R* dx = dinp + n * IC;
    for (int64_t o = 0; o < OC; o++) {
      const R g = dout[n * OC + o];
      const R* wr = W + o * IC;
      for (int64_t i = 0; i < IC; i++) dx[i] += g * wr[i];
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t o = 0; o < OC; o++) {
    R* dw = dW + o * IC;
    for (int64_t n = 0; n < N; n++) {
      const R g = dout[n * OC + o];
      const R* x = inp + n * IC;
      for (int64_t i = 0; i < IC; i++) dw[i] += g * x[i];
    }
    if (dbias) {
      R s = 0;
      for (int64_t n = 0; n < N; n++) s += dout[n * OC + o];
      dbias[o] += s;
    }
  }
}

// Causal multi-head self-attention ([GeekNews] "The Transformer core"):
// q, k, v come from one Linear and are split per head; S = q k^T / sqrt(hs);
// the lower-triangular mask keeps j <= i; softmax over the kept entries;
// y = P v; heads concatenated back in order.
//   qkv row layout: [q (C) | k (C) | v (C)], head h owns channels
//   h*hs .. h*hs+hs-1 of each part.
//   preatt/att: [B, NH, T, T]; masked entries hold -inf / 0.
template <typename R>
void attention_forward(R* out, R* preatt, R* att, const R* qkv, int64_t B,
                       int64_t T, int64_t C, int64_t NH) {
  const int64_t hs = C / NH, C3 = 3 * C;
  const R scale = (R)1 / std::sqrt((R)hs);
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; b++)
    for (int64_t h = 0; h < NH; h++)
      for (int64_t t = 0; t < T; t++) {
        const R* q = qkv + (b * T + t) * C3 + h * hs;
        R* pre = preatt + ((b * NH + h) * T + t) * T;
        R* a = att + ((b * NH + h) * T + t) * T;
        R mx = -std::numeric_limits<R>::infinity();
        for (int64_t t2 = 0; t2 < T; t2++) {
          if (t2 > t) { pre[t2] = -std::numeric_limits<R>::infinity(); continue; }
          const R* k = qkv + (b * T + t2) * C3 + C + h * hs;
          R s = 0;
          for (int64_t i = 0; i < hs; i++) s += q[i] * k[i];
          s = s * scale;
          pre[t2] = s;
          if (s > mx) mx = s;
        }
        R sum = 0;
        for (int64_t t2 = 0; t2 < T; t2++) {
          R e = t2 <= t ? std::exp(pre[t2] - mx) : (R)0;
          a[t2] = e;
          sum += e;
        }
        for (int64_t t2 = 0; t2 < T; t2++) a[t2] = a[t2] / sum;
        R* y = out + (b * T + t) * C + h * hs;
        for (int64_t i = 0; i < hs; i++) y[i] = 0;
        for (int64_t t2 = 0; t2 <= t; t2++) {
          const R* v = qkv + (b * T + t2) * C3 + 2 * C + h * hs;
          for (int64_t i = 0; i < hs; i++) y[i] += a[t2] * v[i];
        }
      }
}

// Attention backward, by the chain rule through y = P v, the softmax and
// S = q k^T * scale:
//   dP = dy v^T;  dv += P^T dy;  dS = P * (dP - rowsum(P * dP));
//   dq += dS k * scale;  dk += dS^T q * scale.
template <typename R>
void attention_backward(R* dqkv, R* dpreatt, R* datt, const R* dout,
                        const R* qkv, const R* att, int64_t B, int64_t T,
                        int64_t C, int64_t NH) {
  const int64_t hs = C / NH, C3 = 3 * C;
  const R scale = (R)1 / std::sqrt((R)hs);
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; b++)
    for (int64_t h = 0; h < NH; h++)
      for (int64_t t = 0; t < T; t++) {
        const R* a = att + ((b * NH + h) * T + t) * T;
        R* da = datt + ((b * NH + h) * T + t) * T;
        R* dpre = dpreatt + ((b * NH + h) * T + t) * T;
        const R* dy = dout + (b * T + t) * C + h * hs;
        for (int64_t t2 = 0; t2 < T; t2++) { da[t2] = 0; dpre[t2] = 0; }
        for (int64_t t2 = 0; t2 <= t; t2++) {
          const R* v = qkv + (b * T + t2) * C3 + 2 * C + h * hs;
          R* dv = dqkv + (b * T + t2) * C3 + 2 * C + h * hs;
          R s = 0;
          for (int64_t i = 0; i < hs; i++) {
            s += dy[i] * v[i];
            dv[i] += a[t2] * dy[i];
          }
          da[t2] = s;
        }
        R pd = 0;
        for (int64_t t2 = 0; t2 <= t; t2++) pd += a[t2] * da[t2];
        for (int64_t t2 = 0; t2 <= t; t2++) dpre[t2] = a[t2] * (da[t2] - pd);
        const R* q = qkv + (b * T + t) * C3 + h * hs;
        R* dq = dqkv + (b * T + t) * C3 + h * hs;
        for (int64_t t2 = 0; t2 <= t; t2++) {
          const R* k = qkv + (b * T + t2) * C3 + C + h * hs;
          R* dk = dqkv + (b * T + t2) * C3 + C + h * hs;
          for (int64_t i = 0; i < hs; i++) {
            dq[i] += dpre[t2] * k[i] * scale;
            dk[i] += dpre[t2] * q[i] * scale;
          }
        }
      }
}

// GELU, tanh form (printed in the [GeekNews] Hacker News comments):
//   gelu(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))).
// sqrt(2/pi) is taken at full precision (the page prints .7978845).
const double kGeluS = 0.79788456080286535588;  // sqrt(2/pi)
const double kGeluA = 0.044715;

template <typename R>
void gelu_forward(R* out, const R* inp, int64_t N) {
  const R s = (R)kGeluS, a = (R)kGeluA;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; i++) {
    const R x = inp[i];
    out[i] = (R)0.5 * x * ((R)1 + std::tanh(s * (x + a * x * x * x)));
  }
}

// d gelu / dx = 1/2 (1 + tanh u) + x/2 (1 - tanh^2 u) sqrt(2/pi) (1 + 3a x^2),
// u = sqrt(2/pi) (x + a x^3).
template <typename R>
void gelu_backward(R* dinp, const R* inp, const R* dout, int64_t N) {
  const R s = (R)kGeluS, a = (R)kGeluA;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; i++) {
    const R x = inp[i];
    const R th = std::tanh(s * (x + a * x * x * x));
    const R d = (R)0.5 * ((R)1 + th) +
                (R)0.5 * x * ((R)1 - th * th) * s * ((R)1 + (R)3 * a * x * x);
    dinp[i] += d * dout[i];
  }
}

// residual connection: out = a + b; the gradient flows unchanged to both.
template <typename R>
void residual_forward(R* out, const R* a, const R* b, int64_t N) {
  for (int64_t i = 0; i < N; i++) out[i] = a[i] + b[i];
}
template <typename R>
void residual_backward(R* da, R* db, const R* dout, int64_t N) {
  for (int64_t i = 0; i < N; i++) { da[i] += dout[i]; db[i] += dout[i]; }
}

// softmax over the V vocabulary entries of each row, and the cross-entropy
// loss of the target ([InfoQ] layer list: softmax, cross-entropy loss):
//   p = exp(l - max l) / sum exp(l - max l);
//   loss = -log p[target] = log(sum exp(l - max l)) - (l[target] - max l).
template <typename R>
void crossentropy_forward(R* losses, R* probs, const R* logits,
                          const int32_t* targets, int64_t N, int64_t V) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; i++) {
    const R* l = logits + i * V;
    R* p = probs + i * V;
    R mx = l[0];
    for (int64_t j = 1; j < V; j++) if (l[j] > mx) mx = l[j];
    R sum = 0;
    for (int64_t j = 0; j < V; j++) { p[j] = std::exp(l[j] - mx); sum += p[j]; }
    for (int64_t j = 0; j < V; j++) p[j] = p[j] / sum;
    if (targets) losses[i] = std::log(sum) - (l[targets[i]] - mx);
  }
}

// d loss_i / d logits_i = p_i - onehot(target_i), times dloss (1/(B*T) for
// the mean).
template <typename R>
void crossentropy_backward(R* dlogits, const R* probs, const int32_t* targets,
                           int64_t N, int64_t V, R dloss) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; i++)
    for (int64_t j = 0; j < V; j++) {
      R ind = j == targets[i] ? (R)1 : (R)0;
      dlogits[i * V + j] += (probs[i * V + j] - ind) * dloss;
    }
}

// AdamW ([InfoQ] "Adam lr 1e-4"; [microgpt] Adam optimiser; decoupled weight
// decay as the plainest reading of a single wd argument):
//   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
//   mhat = m / (1-b1^t);  vhat = v / (1-b2^t);
//   p = p - lr * (mhat / (sqrt(vhat) + eps) + wd * p)
template <typename R>
void adamw_update(int64_t n, R* p, const R* g, R* m, R* v, R lr, R b1, R b2,
                  R eps, R wd, int t) {
  const R c1 = (R)1 - std::pow(b1, (R)t);
  const R c2 = (R)1 - std::pow(b2, (R)t);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) {
    const R mi = b1 * m[i] + ((R)1 - b1) * g[i];
    const R vi = b2 * v[i] + ((R)1 - b2) * g[i] * g[i];
    m[i] = mi;
    v[i] = vi;
    const R mhat = mi / c1;
    const R vhat = vi / c2;
    p[i] = p[i] - lr * (mhat / (std::sqrt(vhat) + eps) + wd * p[i]);
  }
}

// ---------------------------------------------------------------- model

// The whole step, chained layer by layer ([QbitAI]: once every layer has
// its forward and backward, they are strung together).
template <typename R>
struct Model {
  Shape s;
  int64_t psz[NUM_PARAMS], asz[NUM_ACTS];
  std::vector<R> acts, dacts;

  explicit Model(const Shape& sh) : s(sh) {
    param_sizes(s, psz);
    act_sizes(s, asz);
    int64_t na = 0;
    for (int i = 0; i < NUM_ACTS; i++) na += asz[i];
    acts.assign(na, (R)0);
  }

  // Returns the mean loss (NaN when targets == nullptr).
  double forward(const R* params_base, const int32_t* tok, const int32_t* tgt) {
    const int64_t B = s.B, T = s.T, C = s.C, L = s.L, NH = s.NH, BT = B * T;
    Tensors<R> P(const_cast<R*>(params_base), psz, NUM_PARAMS);
    Tensors<R> A(acts.data(), asz, NUM_ACTS);
    encoder_forward(A[ENCODED], tok, P[WTE], P[WPE], B, T, C);
    for (int64_t l = 0; l < L; l++) {
      const R* res = l == 0 ? A[ENCODED] : A[RESIDUAL3] + (l - 1) * BT * C;
      R* ln1 = A[LN1] + l * BT * C;
      R* qkv = A[QKV] + l * BT * 3 * C;
      R* atty = A[ATTY] + l * BT * C;
      R* pre = A[PREATT] + l * B * NH * T * T;
      R* att = A[ATT] + l * B * NH * T * T;
      R* ap = A[ATTPROJ] + l * BT * C;
      R* r2 = A[RESIDUAL2] + l * BT * C;
      R* ln2 = A[LN2] + l * BT * C;
      R* fch = A[FCH] + l * BT * 4 * C;
      R* fcg = A[FCH_GELU] + l * BT * 4 * C;
      R* fp = A[FCPROJ] + l * BT * C;
      R* r3 = A[RESIDUAL3] + l * BT * C;
      layernorm_forward(ln1, A[LN1_MEAN] + l * BT, A[LN1_RSTD] + l * BT, res,
                        P[LN1W] + l * C, P[LN1B] + l * C, BT, C);
      matmul_forward(qkv, ln1, P[QKVW] + l * 3 * C * C, P[QKVB] + l * 3 * C, BT, C, 3 * C);
      attention_forward(atty, pre, att, qkv, B, T, C, NH);
      matmul_forward(ap, atty, P[ATTPROJW] + l * C * C, P[ATTPROJB] + l * C, BT, C, C);
      residual_forward(r2, res, ap, BT * C);
      layernorm_forward(ln2, A[LN2_MEAN] + l * BT, A[LN2_RSTD] + l * BT, r2,
                        P[LN2W] + l * C, P[LN2B] + l * C, BT, C);
      matmul_forward(fch, ln2, P[FCW] + l * 4 * C * C, P[FCB] + l * 4 * C, BT, C, 4 * C);
      gelu_forward(fcg, fch, BT * 4 * C);
      matmul_forward(fp, fcg, P[FCPROJW] + l * 4 * C * C, P[FCPROJB] + l * C, BT, 4 * C, C);
      residual_forward(r3, r2, fp, BT * C);
    }
    const R* last = L == 0 ? A[ENCODED] : A[RESIDUAL3] + (L - 1) * BT * C;
    layernorm_forward(A[LNF], A[LNF_MEAN], A[LNF_RSTD], last, P[LNFW], P[LNFB], BT, C);
    // tied head: the first V rows of wte; pad rows V..Vp-1 take no part.
    matmul_forward(A[LOGITS], A[LNF], P[WTE], (const R*)nullptr, BT, C, s.V);
    crossentropy_forward(A[LOSSES], A[PROBS], A[LOGITS], tgt, BT, s.V);
    if (!tgt) return std::numeric_limits<double>::quiet_NaN();
    double mean = 0;  // the reported scalar; accumulated in double
    for (int64_t i = 0; i < BT; i++) mean += (double)A[LOSSES][i];
    return mean / (double)BT;
  }

  // grads (same layout as params) are overwritten with d(mean loss)/d(param).
  void backward(const R* params_base, R* grads_base, const int32_t* tok,
                const int32_t* tgt) {
    const int64_t B = s.B, T = s.T, C = s.C, L = s.L, NH = s.NH, BT = B * T;
    int64_t np = 0;
    for (int i = 0; i < NUM_PARAMS; i++) np += psz[i];
    std::memset(grads_base, 0, sizeof(R) * np);
    dacts.assign(acts.size(), (R)0);
    Tensors<R> P(const_cast<R*>(params_base), psz, NUM_PARAMS);
    Tensors<R> G(grads_base, psz, NUM_PARAMS);
    Tensors<R> A(acts.data(), asz, NUM_ACTS);
    Tensors<R> D(dacts.data(), asz, NUM_ACTS);
    crossentropy_backward(D[LOGITS], A[PROBS], tgt, BT, s.V, (R)1 / (R)BT);
    matmul_backward(D[LNF], G[WTE], (R*)nullptr, D[LOGITS], A[LNF], P[WTE], BT, C, s.V);
    const R* last = L == 0 ? A[ENCODED] : A[RESIDUAL3] + (L - 1) * BT * C;
    R* dlast = L == 0 ? D[ENCODED] : D[RESIDUAL3] + (L - 1) * BT * C;
    layernorm_backward(dlast, G[LNFW], G[LNFB], D[LNF], last, P[LNFW],
                       A[LNF_MEAN], A[LNF_RSTD], BT, C);
    for (int64_t l = L - 1; l >= 0; l--) {
      const R* res = l == 0 ? A[ENCODED] : A[RESIDUAL3] + (l - 1) * BT * C;
      R* dres = l == 0 ? D[ENCODED] : D[RESIDUAL3] + (l - 1) * BT * C;
      const int64_t o1 = l * BT * C, o3 = l * BT * 3 * C, o4 = l * BT * 4 * C;
      const int64_t oa = l * B * NH * T * T;
      // residual3 = residual2 + fcproj
      residual_backward(D[RESIDUAL2] + o1, D[FCPROJ] + o1, D[RESIDUAL3] + o1, BT * C);
      matmul_backward(D[FCH_GELU] + o4, G[FCPROJW] + l * 4 * C * C, G[FCPROJB] + l * C,
                      D[FCPROJ] + o1, A[FCH_GELU] + o4, P[FCPROJW] + l * 4 * C * C, BT, 4 * C, C);
      gelu_backward(D[FCH] + o4, A[FCH] + o4, D[FCH_GELU] + o4, BT * 4 * C);
      matmul_backward(D[LN2] + o1, G[FCW] + l * 4 * C * C, G[FCB] + l * 4 * C,
                      D[FCH] + o4, A[LN2] + o1, P[FCW] + l * 4 * C * C, BT, C, 4 * C);
      layernorm_backward(D[RESIDUAL2] + o1, G[LN2W] + l * C, G[LN2B] + l * C, D[LN2] + o1,
                         A[RESIDUAL2] + o1, P[LN2W] + l * C, A[LN2_MEAN] + l * BT,
                         A[LN2_RSTD] + l * BT, BT, C);
      // residual2 = residual + attproj
      residual_backward(dres, D[ATTPROJ] + o1, D[RESIDUAL2] + o1, BT * C);
      matmul_backward(D[ATTY] + o1, G[ATTPROJW] + l * C * C, G[ATTPROJB] + l * C,
                      D[ATTPROJ] + o1, A[ATTY] + o1, P[ATTPROJW] + l * C * C, BT, C, C);
      attention_backward(D[QKV] + o3, D[PREATT] + oa, D[ATT] + oa, D[ATTY] + o1,
                         A[QKV] + o3, A[ATT] + oa, B, T, C, NH);
      matmul_backward(D[LN1] + o1, G[QKVW] + l * 3 * C * C, G[QKVB] + l * 3 * C,
                      D[QKV] + o3, A[LN1] + o1, P[QKVW] + l * 3 * C * C, BT, C, 3 * C);
      layernorm_backward(dres, G[LN1W] + l * C, G[LN1B] + l * C, D[LN1] + o1, res,
                         P[LN1W] + l * C, A[LN1_MEAN] + l * BT, A[LN1_RSTD] + l * BT, BT, C);
    }
    encoder_backward(G[WTE], G[WPE], D[ENCODED], tok, B, T, C);
  }
};

template <typename R>
double fwdbwd(const int32_t* cfg8, const R* params, const int32_t* tok,
              const int32_t* tgt, R* grads, R* losses, R* logits) {
  Shape s = shape_from(cfg8);
  if (!shape_ok(s)) return std::numeric_limits<double>::quiet_NaN();
  for (int64_t i = 0; i < s.B * s.T; i++) {
    if (tok[i] < 0 || tok[i] >= s.V) return std::numeric_limits<double>::quiet_NaN();
    if (tgt && (tgt[i] < 0 || tgt[i] >= s.V)) return std::numeric_limits<double>::quiet_NaN();
  }
  Model<R> m(s);
  double loss = m.forward(params, tok, tgt);
  Tensors<R> A(m.acts.data(), m.asz, NUM_ACTS);
  const int64_t BT = s.B * s.T;
  if (losses && tgt) std::memcpy(losses, A[LOSSES], sizeof(R) * BT);
  if (logits) std::memcpy(logits, A[LOGITS], sizeof(R) * BT * s.V);
  if (grads && tgt) m.backward(params, grads, tok, tgt);
  return loss;
}

// ---------------------------------------------------------------- generation

// One new position `pos` of one sequence, computed with a key/value cache
// ([GeekNews], "How KV caching works": after a token is generated the next
// one needs only the new row; the keys and values of the earlier rows are
// kept from the earlier iterations and reused).  kc, vc: this sequence's
// cache, [L][maxT][C]; rows 0..pos-1 hold the earlier positions and row pos
// is written here.  The arithmetic of every step is the one of the full
// forward above, applied to the single new row; the attention of the new
// query over cache rows 0..pos is the row t = pos of attention_forward.
// logits: the V scores of the new row ([GeekNews], "The Transformer core":
// the final LayerNorm output at the last position times the embedding
// matrix).
template <typename R>
void decode_position(const Shape& s, const R* params, R* kc, R* vc, int32_t token, int64_t pos,
                     R* logits) {
  const int64_t C = s.C, L = s.L, NH = s.NH, hs = C / NH, maxT = s.maxT;
  int64_t psz[NUM_PARAMS];
  param_sizes(s, psz);
  Tensors<R> P(const_cast<R*>(params), psz, NUM_PARAMS);
  std::vector<R> x(C), ln(C), qkv(3 * C), y(C), ap(C), x2(C), fch(4 * C), fcg(4 * C), fp(C);
  std::vector<R> sc(pos + 1);
  R mean = 0, rstd = 0;
  // token embedding plus the embedding of position pos
  encoder_forward(x.data(), &token, P[WTE], P[WPE] + pos * C, 1, 1, C);
  const R scale = (R)1 / std::sqrt((R)hs);
  for (int64_t l = 0; l < L; l++) {
    R* kl = kc + l * maxT * C;
    R* vl = vc + l * maxT * C;
    layernorm_forward(ln.data(), &mean, &rstd, x.data(), P[LN1W] + l * C, P[LN1B] + l * C, 1, C);
    matmul_forward(qkv.data(), ln.data(), P[QKVW] + l * 3 * C * C, P[QKVB] + l * 3 * C, 1, C, 3 * C);
    for (int64_t i = 0; i < C; i++) {
      kl[pos * C + i] = qkv[C + i];
      vl[pos * C + i] = qkv[2 * C + i];
    }
    for (int64_t h = 0; h < NH; h++) {
      const R* q = qkv.data() + h * hs;
      R mx = -std::numeric_limits<R>::infinity();
      for (int64_t j = 0; j <= pos; j++) {
        const R* k = kl + j * C + h * hs;
        R d = 0;
        for (int64_t i = 0; i < hs; i++) d += q[i] * k[i];
        d = d * scale;
        sc[j] = d;
        if (d > mx) mx = d;
      }
      R sum = 0;
      for (int64_t j = 0; j <= pos; j++) {
        sc[j] = std::exp(sc[j] - mx);
        sum += sc[j];
      }
      for (int64_t j = 0; j <= pos; j++) sc[j] = sc[j] / sum;
      R* yh = y.data() + h * hs;
      for (int64_t i = 0; i < hs; i++) yh[i] = 0;
      for (int64_t j = 0; j <= pos; j++) {
        const R* v = vl + j * C + h * hs;
        for (int64_t i = 0; i < hs; i++) yh[i] += sc[j] * v[i];
      }
    }
    matmul_forward(ap.data(), y.data(), P[ATTPROJW] + l * C * C, P[ATTPROJB] + l * C, 1, C, C);
    residual_forward(x2.data(), x.data(), ap.data(), C);
    layernorm_forward(ln.data(), &mean, &rstd, x2.data(), P[LN2W] + l * C, P[LN2B] + l * C, 1, C);
    matmul_forward(fch.data(), ln.data(), P[FCW] + l * 4 * C * C, P[FCB] + l * 4 * C, 1, C, 4 * C);
    gelu_forward(fcg.data(), fch.data(), 4 * C);
    matmul_forward(fp.data(), fcg.data(), P[FCPROJW] + l * 4 * C * C, P[FCPROJB] + l * C, 1, 4 * C, C);
    residual_forward(x.data(), x2.data(), fp.data(), C);
  }
  layernorm_forward(ln.data(), &mean, &rstd, x.data(), P[LNFW], P[LNFB], 1, C);
  matmul_forward(logits, ln.data(), P[WTE], (const R*)nullptr, 1, C, s.V);
}

// The next token drawn from the V scores of one row.  The pages print the
// generated ids ([InfoQ] run log, "generated: ...") but not the rule; the
// plainest reading taken here is inverse-CDF sampling of the softmax at a
// temperature: p_i proportional to exp((l_i - max l) / temperature), and
// the token is the smallest i whose running sum p_0 + ... + p_i exceeds
// u * (p_0 + ... + p_{V-1}), u a uniform draw in [0, 1) supplied by the
// caller.  temperature <= 0 is greedy decoding: the first index of the
// largest score.  Should rounding leave no running sum above the threshold,
// the last index with p_i > 0 is taken.
int64_t sample_row(const double* l, int64_t V, double temperature, double u) {
  int64_t best = 0;
  for (int64_t i = 1; i < V; i++) if (l[i] > l[best]) best = i;
  if (!(temperature > 0)) return best;
  const double mx = l[best];
  std::vector<double> p(V);
  double sum = 0;
  for (int64_t i = 0; i < V; i++) {
    p[i] = std::exp((l[i] - mx) / temperature);
    sum += p[i];
  }
  const double target = u * sum;
  double run = 0;
  int64_t last = best;
  for (int64_t i = 0; i < V; i++) {
    run += p[i];
    if (p[i] > 0) last = i;
    if (run > target) return i;
  }
  return last;
}

// ---------------------------------------------------------------- FP8 (E4M3)
// Lower precision for the matmuls ([QbitAI]: precision can go from fp32 to
// fp16 or lower).  The 8-bit format is E4M3 as the OCP FP8 specification
// defines it: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; a
// code with exponent field e > 0 is (-1)^s 2^(e-7) (1 + m/8), with e = 0 it
// is (-1)^s 2^-6 (m/8) (subnormal); S.1111.111 is NaN; there is no infinity,
// so the largest finite magnitude is 2^8 * 1.75 = 448.
double e4m3_decode(uint8_t c) {
  const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = e == 0 ? std::ldexp((double)m / 8.0, -6) : std::ldexp(1.0 + (double)m / 8.0, e - 7);
  return sgn ? -mag : mag;
}

// The code nearest to x (ties to the code with an even mantissa field, i.e.
// round-half-to-even on the 3-bit mantissa grid); magnitudes above 448
// saturate to 448 (the "satfinite" conversion); NaN gives NaN.  Written as a
// search over the 127 non-negative finite codes, which are in increasing
// order of value.
uint8_t e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sgn = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  if (a >= 448.0) return sgn | 0x7E;
  uint8_t lo = 0;  // largest code with value <= a
  for (int c = 1; c <= 0x7E; c++)
    if (e4m3_decode((uint8_t)c) <= a) lo = (uint8_t)c;
  const uint8_t hi = (uint8_t)(lo + 1);
  const double dl = a - e4m3_decode(lo), dh = e4m3_decode(hi) - a;
  uint8_t c = lo;
  if (dh < dl || (dh == dl && (hi & 1) == 0)) c = hi;
  return sgn | c;
}

// Per-tensor scaling: s = 448 / max|x| (1 when x is all zeros) maps the
// largest magnitude onto the largest code; q_i = encode(x_i * s) with the
// product taken in float, as a float32 pipeline computes it.
float fp8_quantize(const float* x, int64_t n, uint8_t* q) {
  float amax = 0.f;
  for (int64_t i = 0; i < n; i++) amax = std::fmax(amax, std::fabs(x[i]));
  const float s = amax > 0.f ? 448.f / amax : 1.f;
  for (int64_t i = 0; i < n; i++) q[i] = e4m3_encode((double)(x[i] * s));
  return s;
}

// out[m, n] = (sum_k dec(qa[m, k]) dec(qb[n, k])) / (sa sb) (+ bias[n]):
// the matmul of the two dequantised operands, in double.
void fp8_matmul(double* out, const uint8_t* qa, double sa, const uint8_t* qb, double sb,
                const double* bias, int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; m++)
    for (int64_t n = 0; n < N; n++) {
      double acc = 0;
      for (int64_t k = 0; k < K; k++) acc += e4m3_decode(qa[m * K + k]) * e4m3_decode(qb[n * K + k]);
      out[m * N + n] = acc / (sa * sb) + (bias ? bias[n] : 0.0);
    }
}

// ---------------------------------------------------------------- init RNG

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
// published multipliers and Weyl key increments.
void philox4x32_10(const uint32_t in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = in[0], c1 = in[1], c2 = in[2], c3 = in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; r++) {
    if (r > 0) { k0 += W0; k1 += W1; }
    const uint64_t p0 = (uint64_t)M0 * c0;
    const uint64_t p1 = (uint64_t)M1 * c2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// Standard normal draw for arena element e: Philox block at counter
// (e/2, 0, 0) under key = seed; words 0 and 1 become u1 = (x0+1)/2^32 in
// (0,1] and u2 = x1/2^32 in [0,1); Box-Muller gives r cos(2 pi u2) for even e
// and r sin(2 pi u2) for odd e, r = sqrt(-2 ln u1).
double normal_at(uint64_t seed, int64_t e) {
  const uint64_t pair = (uint64_t)e >> 1;
  const uint32_t ctr[4] = {(uint32_t)pair, (uint32_t)(pair >> 32), 0u, 0u};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t x[4];
  philox4x32_10(ctr, key, x);
  const double u1 = ((double)x[0] + 1.0) / 4294967296.0;
  const double u2 = (double)x[1] / 4294967296.0;
  const double r = std::sqrt(-2.0 * std::log(u1));
  const double th = 6.283185307179586476925 * u2;
  return (e & 1) ? r * std::sin(th) : r * std::cos(th);
}

}  // namespace

// ---------------------------------------------------------------- C surface

extern "C" {

int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

int64_t oracle_num_params(const int32_t* cfg8) {
  Shape s = shape_from(cfg8);
  int64_t n[NUM_PARAMS], t = 0;
  param_sizes(s, n);
  for (int i = 0; i < NUM_PARAMS; i++) t += n[i];
  return t;
}

int64_t oracle_num_activations(const int32_t* cfg8) {
  Shape s = shape_from(cfg8);
  int64_t n[NUM_ACTS], t = 0;
  act_sizes(s, n);
  for (int i = 0; i < NUM_ACTS; i++) t += n[i];
  return t;
}

int oracle_num_param_tensors(void) { return NUM_PARAMS; }

// offset and size of parameter tensor idx inside the 1-D parameter array.
int oracle_param_tensor(const int32_t* cfg8, int idx, int64_t* offset, int64_t* numel) {
  if (idx < 0 || idx >= NUM_PARAMS) return -1;
  Shape s = shape_from(cfg8);
  int64_t n[NUM_PARAMS], off = 0;
  param_sizes(s, n);
  for (int i = 0; i < idx; i++) off += n[i];
  *offset = off;
  *numel = n[idx];
  return 0;
}

void oracle_philox4x32_10(const uint32_t* ctr4, const uint32_t* key2, uint32_t* out4) {
  philox4x32_10(ctr4, key2, out4);
}

double oracle_normal_at(uint64_t seed, int64_t e) { return normal_at(seed, e); }

// The initial parameters the library's build step is specified to draw:
// N(0, 0.02) for wte rows < V, wpe and the four Linear weights, the two
// residual projections (attproj, fcproj) further scaled by 1/sqrt(2L);
// biases 0, LayerNorm gamma 1 and beta 0; wte pad rows 0.
int oracle_init_params(const int32_t* cfg8, uint64_t seed, double* out) {
  Shape s = shape_from(cfg8);
  if (!shape_ok(s)) return -1;
  int64_t n[NUM_PARAMS];
  param_sizes(s, n);
  const double sd = 0.02, sdr = 0.02 / std::sqrt(2.0 * (double)(s.L > 0 ? s.L : 1));
  int64_t off = 0;
  for (int t = 0; t < NUM_PARAMS; t++) {
    for (int64_t i = 0; i < n[t]; i++) {
      const int64_t e = off + i;
      double v = 0.0;
      switch (t) {
        case WTE: v = (i / s.C) < s.V ? sd * normal_at(seed, e) : 0.0; break;
        case WPE: case QKVW: case FCW: v = sd * normal_at(seed, e); break;
        case ATTPROJW: case FCPROJW: v = sdr * normal_at(seed, e); break;
        case LN1W: case LN2W: case LNFW: v = 1.0; break;
        default: v = 0.0; break;
      }
      out[e] = v;
    }
    off += n[t];
  }
  return 0;
}

// One forward (+ backward when grads and targets are given) of the whole
// model.  grads are overwritten (not accumulated).  losses: [B*T];
// logits: [B*T, V] (unpadded).  Any output pointer may be null.
double oracle_fwdbwd_f32(const int32_t* cfg8, const float* params, const int32_t* tok,
                         const int32_t* tgt, float* grads, float* losses, float* logits) {
  return fwdbwd<float>(cfg8, params, tok, tgt, grads, losses, logits);
}
// The residual streams of a forward pass: out[(L+1), B*T, C]; stream 0 is the
// encoder output, stream l the output of block l-1.
int oracle_residuals_f32(const int32_t* cfg8, const float* params, const int32_t* tok, float* out) {
  Shape s = shape_from(cfg8);
  if (!shape_ok(s)) return -1;
  Model<float> m(s);
  m.forward(params, tok, nullptr);
  Tensors<float> A(m.acts.data(), m.asz, NUM_ACTS);
  const int64_t n = s.B * s.T * s.C;
  std::memcpy(out, A[ENCODED], sizeof(float) * n);
  for (int64_t l = 0; l < s.L; l++) std::memcpy(out + (l + 1) * n, A[RESIDUAL3] + l * n, sizeof(float) * n);
  return 0;
}
double oracle_fwdbwd_f64(const int32_t* cfg8, const double* params, const int32_t* tok,
                         const int32_t* tgt, double* grads, double* losses, double* logits) {
  return fwdbwd<double>(cfg8, params, tok, tgt, grads, losses, logits);
}

// Logits of every position of tok [B, T], computed position by position with
// the key/value cache of decode_position (row t of sequence b uses cache rows
// 0..t).  out: [B, T, V].  Returns 0, or -1 for a bad shape or id.
int oracle_decode_logits_f64(const int32_t* cfg8, const double* params, const int32_t* tok,
                             double* out) {
  Shape s = shape_from(cfg8);
  if (!shape_ok(s) || s.T > s.maxT) return -1;
  for (int64_t i = 0; i < s.B * s.T; i++)
    if (tok[i] < 0 || tok[i] >= s.V) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < s.B; b++) {
    std::vector<double> kc(s.L * s.maxT * s.C), vc(s.L * s.maxT * s.C);
    for (int64_t t = 0; t < s.T; t++)
      decode_position(s, params, kc.data(), vc.data(), tok[b * s.T + t], t, out + (b * s.T + t) * s.V);
  }
  return 0;
}

// Generation: for each of the B sequences, the prompt prompt[b, 0..T0-1] is
// run through decode_position (filling the cache), then n_new tokens are
// drawn one at a time with sample_row from the scores of the last row, the
// drawn token being the input of the next position.  uniforms: [n_new, B],
// the draw of new token i of sequence b at uniforms[i * B + b].
// out_tokens: [B, T0 + n_new] (prompt, then the drawn tokens); out_logits
// (may be null): [n_new, B, V], the scores each new token was drawn from.
// Needs 1 <= T0 and T0 + n_new <= maxT + 1 (the last drawn token is not fed
// back).  Returns 0, or -1 for a bad shape or id.
int oracle_generate_f64(const int32_t* cfg8, const double* params, const int32_t* prompt, int64_t T0,
                        int64_t n_new, double temperature, const double* uniforms, int32_t* out_tokens,
                        double* out_logits) {
  Shape s = shape_from(cfg8);
  if (!shape_ok(s) || T0 < 1 || n_new < 0 || T0 + n_new > s.maxT + 1 || T0 > s.maxT) return -1;
  for (int64_t i = 0; i < s.B * T0; i++)
    if (prompt[i] < 0 || prompt[i] >= s.V) return -1;
  const int64_t TT = T0 + n_new;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < s.B; b++) {
    std::vector<double> kc(s.L * s.maxT * s.C), vc(s.L * s.maxT * s.C), lg(s.V);
    for (int64_t t = 0; t < T0; t++) out_tokens[b * TT + t] = prompt[b * T0 + t];
    for (int64_t t = 0; t < T0 - 1; t++)
      decode_position(s, params, kc.data(), vc.data(), prompt[b * T0 + t], t, lg.data());
    int32_t cur = prompt[b * T0 + T0 - 1];
    for (int64_t i = 0; i < n_new; i++) {
      decode_position(s, params, kc.data(), vc.data(), cur, T0 - 1 + i, lg.data());
      if (out_logits) std::memcpy(out_logits + (i * s.B + b) * s.V, lg.data(), sizeof(double) * s.V);
      cur = (int32_t)sample_row(lg.data(), s.V, temperature, uniforms[i * s.B + b]);
      out_tokens[b * TT + T0 + i] = cur;
    }
  }
  return 0;
}

int64_t oracle_sample_f64(const double* logits, int64_t V, double temperature, double u) {
  return sample_row(logits, V, temperature, u);
}

double oracle_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
uint8_t oracle_e4m3_encode(double x) { return e4m3_encode(x); }
float oracle_fp8_quantize(const float* x, int64_t n, uint8_t* q) { return fp8_quantize(x, n, q); }
void oracle_fp8_matmul(double* out, const uint8_t* qa, double sa, const uint8_t* qb, double sb,
                       const double* bias, int64_t M, int64_t N, int64_t K) {
  fp8_matmul(out, qa, sa, qb, sb, bias, M, N, K);
}

void oracle_adamw_f32(int64_t n, float* p, const float* g, float* m, float* v, float lr,
                      float b1, float b2, float eps, float wd, int t) {
  adamw_update<float>(n, p, g, m, v, lr, b1, b2, eps, wd, t);
}
void oracle_adamw_f64(int64_t n, double* p, const double* g, double* m, double* v, double lr,
                      double b1, double b2, double eps, double wd, int t) {
  adamw_update<double>(n, p, g, m, v, lr, b1, b2, eps, wd, t);
}

// Layer primitives in double, exposed for the pins.
void oracle_encoder_forward_f64(double* out, const int32_t* tok, const double* wte,
                                const double* wpe, int64_t B, int64_t T, int64_t C) {
  encoder_forward(out, tok, wte, wpe, B, T, C);
}
void oracle_encoder_backward_f64(double* dwte, double* dwpe, const double* dout,
                                 const int32_t* tok, int64_t B, int64_t T, int64_t C) {
  encoder_backward(dwte, dwpe, dout, tok, B, T, C);
}
void oracle_layernorm_forward_f64(double* out, double* mean, double* rstd, const double* inp,
                                  const double* w, const double* b, int64_t N, int64_t C) {
  layernorm_forward(out, mean, rstd, inp, w, b, N, C);
}
void oracle_layernorm_backward_f64(double* dinp, double* dw, double* db, const double* dout,
                                   const double* inp, const double* w, const double* mean,
                                   const double* rstd, int64_t N, int64_t C) {
  layernorm_backward(dinp, dw, db, dout, inp, w, mean, rstd, N, C);
}
void oracle_matmul_forward_f64(double* out, const double* inp, const double* W,
                               const double* bias, int64_t N, int64_t IC, int64_t OC) {
  matmul_forward(out, inp, W, bias, N, IC, OC);
}
void oracle_matmul_backward_f64(double* dinp, double* dW, double* dbias, const double* dout,
                                const double* inp, const double* W, int64_t N, int64_t IC,
                                int64_t OC) {
  matmul_backward(dinp, dW, dbias, dout, inp, W, N, IC, OC);
}
void oracle_attention_forward_f64(double* out, double* preatt, double* att, const double* qkv,
                                  int64_t B, int64_t T, int64_t C, int64_t NH) {
  attention_forward(out, preatt, att, qkv, B, T, C, NH);
}
void oracle_attention_backward_f64(double* dqkv, double* dpreatt, double* datt,
                                   const double* dout, const double* qkv, const double* att,
                                   int64_t B, int64_t T, int64_t C, int64_t NH) {
  attention_backward(dqkv, dpreatt, datt, dout, qkv, att, B, T, C, NH);
}
void oracle_gelu_forward_f64(double* out, const double* inp, int64_t N) {
  gelu_forward(out, inp, N);
}
void oracle_gelu_backward_f64(double* dinp, const double* inp, const double* dout, int64_t N) {
  gelu_backward(dinp, inp, dout, N);
}
void oracle_crossentropy_forward_f64(double* losses, double* probs, const double* logits,
                                     const int32_t* tgt, int64_t N, int64_t V) {
  crossentropy_forward(losses, probs, logits, tgt, N, V);
}
void oracle_crossentropy_backward_f64(double* dlogits, const double* probs, const int32_t* tgt,
                                      int64_t N, int64_t V, double dloss) {
  crossentropy_backward(dlogits, probs, tgt, N, V, dloss);
}

}  // extern "C"
