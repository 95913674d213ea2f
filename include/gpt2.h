/*
 * gpt2.h -- C ABI of the B300-native GPT-2 training step (libgpt2.so).
 *
 * The library computes one GPT-2 training step -- forward pass with the
 * mean cross-entropy loss, backward pass, AdamW update -- over memory it
 * allocates once at build time, the design of llm.c as described in
 * QbitAI, "OpenAI founder hand-writes a thousand lines of C to train GPT"
 * (section "Manually implementing each layer's forward/backward pass": all
 * memory is allocated at the start as one 1-D block and stays constant while
 * batches stream through) and in InfoQ, "Real men program in C: a large
 * model hand-built from 1000 lines of C" (the layer list: encoder,
 * layernorm, matmul, self-attention, gelu, residual, softmax, cross-entropy;
 * the forward / zero-grad / backward / update loop).
 *
 * Every stage runs in the library's own sm_103a CUDA kernels.  There is no
 * CPU fallback: a call that cannot run on the GPU returns an error.
 *
 * Conventions for every function below
 *   - Return value: GPT2_OK (0) or one of the negative GPT2_ERR_* codes.
 *     No function aborts, throws or traps; gpt2_last_error() gives text.
 *   - A gpt2_model is used by one host thread at a time; calls are not
 *     re-entrant.  Work is enqueued on the model's stream (gpt2_set_stream)
 *     and is asynchronous unless the function says it synchronises.
 *   - "device pointer" = CUDA global memory on the model's device;
 *     "host pointer" = ordinary (optionally pinned) host memory.
 *   - All floating-point tensors are row-major and contiguous.
 */
#ifndef GPT2_H
#define GPT2_H

#include <stdint.h>

#if defined(__GNUC__)
#define GPT2_API __attribute__((visibility("default")))
#else
#define GPT2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ codes */
#define GPT2_OK 0
#define GPT2_ERR_ARG (-1)       /* null pointer, bad shape, bad argument value    */
#define GPT2_ERR_OOM (-2)       /* a device allocation at build time failed       */
#define GPT2_ERR_CUDA (-3)      /* a CUDA runtime/driver call failed              */
#define GPT2_ERR_STATE (-4)     /* call-order violation (e.g. backward w/o loss)  */
#define GPT2_ERR_TOKEN (-5)     /* a token or target id outside [0, V)            */
#define GPT2_ERR_TIMEOUT (-6)   /* a bounded device-side wait expired             */
#define GPT2_ERR_NONFINITE (-7) /* the loss is NaN or infinite                    */
#define GPT2_ERR_IO (-8)        /* a checkpoint or token file could not be read,
                                   written, or is truncated                      */

/* Arithmetic of the step.
 *   GPT2_FP32: every product and sum in fp32 (SIMT FFMA; no TF32, no bf16).
 *   GPT2_BF16: fp32 master weights, Adam moments and gradients; the matmul and
 *              attention operands are bf16 (a bf16 copy of the weights is
 *              refreshed by every AdamW step) with fp32 accumulation on the
 *              tcgen05 tensor cores; the residual stream, LayerNorm
 *              statistics, softmax statistics and losses stay fp32. */
typedef enum { GPT2_FP32 = 0, GPT2_BF16 = 1 } gpt2_precision;

/* Model shape and the batch shape the buffers are sized for.  The fields
 * named after the run log's header block (max_seq_len, vocab_size,
 * num_layers, num_heads, channels) mean what they mean there.
 * Constraints (checked by gpt2_build, GPT2_ERR_ARG otherwise):
 *   num_layers >= 1; 8 <= channels <= 1024 (the LayerNorm kernels keep a
 *   row's per-column partial sums in registers); channels % num_heads == 0;
 *   channels % 8 == 0;
 *   head size channels/num_heads in {16, 32, 64, 128};
 *   vocab_size <= padded_vocab_size and padded_vocab_size % 8 == 0;
 *   padded_vocab_size <= 262144 (token ids fit 18 bits);
 *   1 <= seq_len <= max_seq_len <= 4096; batch_size >= 1;
 *   batch_size * seq_len <= 32768;
 *   padded_vocab_size * batch_size * seq_len < 2^32. */
typedef struct gpt2_config {
  int32_t max_seq_len;       /* maxT: rows of the position embedding          */
  int32_t vocab_size;        /* V: real vocabulary, the softmax's width       */
  int32_t padded_vocab_size; /* Vp: rows of the token embedding (pad rows 0)  */
  int32_t num_layers;        /* L                                              */
  int32_t num_heads;         /* NH                                             */
  int32_t channels;          /* C                                              */
  int32_t batch_size;        /* B                                              */
  int32_t seq_len;           /* T                                              */
  int32_t precision;         /* gpt2_precision                                 */
} gpt2_config;

/* Opaque model: owns every device buffer (parameter, gradient, AdamW m and
 * v arrays, the bf16 weight copy, the activations, the scratch). */
typedef struct gpt2_model gpt2_model;

/* The four fp32 arrays that share the parameter layout (gpt2_tensor_info). */
typedef enum {
  GPT2_PARAMS = 0, GPT2_GRADS = 1, GPT2_ADAM_M = 2, GPT2_ADAM_V = 3
} gpt2_arena;

/* Allocate every buffer once on the current CUDA device and draw the
 * initial parameters on the device:
 *   N(0, 0.02) for wte rows < V, wpe and the qkv / attproj / fc / fcproj
 *   weights, attproj and fcproj further scaled by 1/sqrt(2 L); all biases 0;
 *   LayerNorm gamma 1, beta 0; wte pad rows 0.
 * The normal draw for parameter-array element e: Philox4x32-10 (Salmon et
 * al., SC'11) at counter (e/2 low word, e/2 high word, 0, 0), key (seed low
 * word, seed high word); u1 = (word0 + 1) / 2^32, u2 = word1 / 2^32;
 * sqrt(-2 ln u1) * cos(2 pi u2) for even e, * sin(2 pi u2) for odd e.
 * Gradients and Adam moments start at zero.  Synchronises.
 *   cfg: host pointer, read only during the call.
 *   out: host pointer that receives the model (NULL on failure).
 * Errors: GPT2_ERR_ARG (bad shape), GPT2_ERR_OOM, GPT2_ERR_CUDA. */
GPT2_API int gpt2_build(const gpt2_config* cfg, uint64_t seed, gpt2_model** out);

/* Release every buffer of the model; NULL is allowed.  Synchronises. */
GPT2_API void gpt2_free(gpt2_model* m);

/* Enqueue all later work on this stream (a cudaStream_t, e.g. a torch
 * stream's handle; NULL = the legacy default stream).  The caller keeps the
 * stream alive while the model uses it. */
GPT2_API int gpt2_set_stream(gpt2_model* m, void* cuda_stream);

/* Forward pass over one batch.
 *   tokens:  device pointer, int32 [B, T], ids in [0, V).
 *   targets: device pointer, int32 [B, T] next-token ids in [0, V), or NULL
 *            for logits only (then gpt2_backward returns GPT2_ERR_STATE and
 *            gpt2_copy_logits_out becomes valid).
 *   mean_loss: host pointer or NULL.  If non-NULL the call synchronises and
 *            writes the mean over the B*T positions of -log softmax(logits)
 *            [target]; it then also reports device-side errors (out-of-range
 *            ids: GPT2_ERR_TOKEN; NaN/Inf loss: GPT2_ERR_NONFINITE).  If NULL
 *            the call is asynchronous; errors surface at the next
 *            synchronising call.
 * The ids are copied into the model, so the caller may reuse the buffers
 * once the stream has passed this call.  With targets, the softmax-minus-
 * one-hot gradient of the loss is computed in the same pass, ready for
 * gpt2_backward. */
GPT2_API int gpt2_forward(gpt2_model* m, const int32_t* tokens, const int32_t* targets,
                 float* mean_loss);

/* As gpt2_forward, with tokens and targets in host memory (pinned memory
 * makes the copy asynchronous); the host-to-device copies are enqueued on
 * the model's stream before the forward pass. */
GPT2_API int gpt2_forward_host(gpt2_model* m, const int32_t* host_tokens,
                      const int32_t* host_targets, float* mean_loss);

/* Set every gradient to zero (the gradient array is accumulated into). */
GPT2_API int gpt2_zero_grad(gpt2_model* m);

/* Backward pass of the last forward (which must have had targets):
 * gradients of the mean loss with respect to every parameter are ADDED to
 * the gradient array.  Asynchronous. */
GPT2_API int gpt2_backward(gpt2_model* m);

/* One AdamW update of every parameter, t = 1-based step number:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p = p - lr * ( (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + wd * p ).
 * Also refreshes the bf16 weight copy (bf16 mode).  Asynchronous.
 * Errors: GPT2_ERR_ARG for t < 1 or a non-finite hyper-parameter. */
GPT2_API int gpt2_adamw_step(gpt2_model* m, float lr, float beta1, float beta2,
                    float eps, float weight_decay, int32_t t);

/* Wait for all enqueued work; report device-side errors recorded since the
 * last synchronising call (GPT2_ERR_TOKEN, GPT2_ERR_TIMEOUT). */
GPT2_API int gpt2_synchronize(gpt2_model* m);

/* Failure-path check of the bounded device waits: enqueues, on the model's
 * stream, one kernel that waits on an mbarrier that nothing ever completes,
 * with the same time limit as every wait of the library's kernels (2 s).
 * The wait gives up, the kernel ends normally, and the next synchronising
 * call reports GPT2_ERR_TIMEOUT and clears the condition; the model stays
 * usable.  For tests of the error path: no fault, trap or hang is involved.
 * Errors: GPT2_ERR_ARG (NULL model), GPT2_ERR_CUDA (launch failed). */
GPT2_API int gpt2_expire_a_wait(gpt2_model* m);

/* The configuration the model was built with. */
GPT2_API int gpt2_get_config(const gpt2_model* m, gpt2_config* out);

/* Number of fp32 elements in the parameter array (Vp rows of wte). */
GPT2_API int gpt2_num_params(const gpt2_model* m, int64_t* n);

/* Number of parameter tensors (16) and, for 0 <= idx < that number, the
 * name, element offset and element count of tensor idx in the parameter
 * array.  Order: wte[Vp,C], wpe[maxT,C], ln1w[L,C], ln1b[L,C],
 * qkvw[L,3C,C], qkvb[L,3C], attprojw[L,C,C], attprojb[L,C], ln2w[L,C],
 * ln2b[L,C], fcw[L,4C,C], fcb[L,4C], fcprojw[L,C,4C], fcprojb[L,C],
 * lnfw[C], lnfb[C].  A Linear's weight is [out, in]: y = x W^T + b.
 * *name points to static storage. */
GPT2_API int gpt2_num_tensors(const gpt2_model* m, int32_t* n);
GPT2_API int gpt2_tensor_info(const gpt2_model* m, int32_t idx, const char** name,
                     int64_t* offset, int64_t* numel);

/* Copy one fp32 array (gpt2_arena) out to / in from host memory of
 * gpt2_num_params floats.  Synchronises.  Copying parameters in also
 * refreshes the bf16 weight copy. */
GPT2_API int gpt2_copy_out(gpt2_model* m, int32_t arena, float* host_dst);
GPT2_API int gpt2_copy_in(gpt2_model* m, int32_t arena, const float* host_src);
/* The same for one named array each: gpt2_copy_params_out(m, dst) is
 * gpt2_copy_out(m, GPT2_PARAMS, dst), and so on for the gradients and the
 * AdamW moments; gpt2_copy_params_in(m, src) is gpt2_copy_in(m,
 * GPT2_PARAMS, src). */
GPT2_API int gpt2_copy_params_out(gpt2_model* m, float* host_dst);
GPT2_API int gpt2_copy_grads_out(gpt2_model* m, float* host_dst);
GPT2_API int gpt2_copy_m_out(gpt2_model* m, float* host_dst);
GPT2_API int gpt2_copy_v_out(gpt2_model* m, float* host_dst);
GPT2_API int gpt2_copy_params_in(gpt2_model* m, const float* host_src);
/* *out = the device address of the fp32 mean loss that a gpt2_forward with
 * targets writes (valid for the model's lifetime; read it in the model's
 * stream order, e.g. after gpt2_forward(..., NULL) without a host sync).
 * Errors: GPT2_ERR_ARG for a NULL model or out. */
GPT2_API int gpt2_loss_device_ptr(const gpt2_model* m, const float** out);

/* Per-position losses [B*T] of the last forward with targets.  Synchronises. */
GPT2_API int gpt2_copy_losses_out(gpt2_model* m, float* host_dst);

/* Logits [B*T, Vp] (as fp32; pad columns are 0 * lnf = 0) of the last
 * forward WITHOUT targets.  Synchronises.  GPT2_ERR_STATE otherwise. */
GPT2_API int gpt2_copy_logits_out(gpt2_model* m, float* host_dst);

/* The fp32 residual stream [B*T, C] entering block `layer` of the last
 * forward: layer 0 is the encoder output wte[token] + wpe[position],
 * layer L the input of the final LayerNorm.  Synchronises.
 * Errors: GPT2_ERR_ARG (layer outside [0, L]), GPT2_ERR_STATE (no forward). */
GPT2_API int gpt2_copy_residual_out(gpt2_model* m, int32_t layer, float* host_dst);

/* Mean loss of the last forward with targets, copied to host memory.
 * Synchronises; reports device-side errors like gpt2_synchronize and
 * GPT2_ERR_NONFINITE for a NaN/Inf loss. */
GPT2_API int gpt2_read_loss(gpt2_model* m, float* host_loss);

/* ---------------------------------------------------------------- generation
 * Decoding with a key/value cache.  GeekNews, "A GPT-2-based ChatGPT clone in
 * 3000 bytes of C", section "How KV caching works": after a token is
 * generated, the results of the earlier rows are reused and only the new row
 * is computed; section "The Transformer core": the final LayerNorm output at
 * the last position times the embedding matrix scores the next token.  The
 * cache is the per-layer qkv activation of gpt2_forward ([B, T, 3C] per
 * layer, in the model's activation precision): a gpt2_forward over a batch
 * whose first P positions are the prompts fills rows 0..P-1 (later rows do
 * not influence them: attention is causal), then one gpt2_decode_step per
 * new position pos = P-1+i ... appends.
 *
 * gpt2_decode_step computes position pos of every sequence b: the input id
 * tokens[b] (device, [B] int32) at position pos; keys and values of that
 * row are written into row pos of the cache, its query attends to rows
 * 0..pos (the caller guarantees rows 0..pos-1 hold this sequence's earlier
 * positions); the scores l of the row (its V real columns) give
 * next_tokens[b] (device, [B] int32): the smallest i whose running sum of
 * p_j = exp((l_j - max l) / temperature) passes uniforms[b] * sum_j p_j
 * (inverse-CDF sampling; uniforms: device [B] floats in [0, 1) that the
 * caller draws), or, for temperature <= 0, the first index of the largest
 * score.  All three pointers are read / written on the model's stream
 * after the call returns (stream order); the caller owns them.  A row pos
 * and its input can be fed back as tokens = next_tokens for pos + 1.
 * Asynchronous: errors of the device side (an id outside [0, V)) surface at
 * the next synchronising call.  After a decode step the training state of
 * the last forward is gone (gpt2_backward needs a new gpt2_forward);
 * gpt2_adamw_step, gpt2_copy_in(GPT2_PARAMS) and gpt2_load_checkpoint
 * invalidate the cache.  Errors: GPT2_ERR_ARG (NULL pointer, pos outside
 * [0, T), non-finite temperature), GPT2_ERR_STATE (no cache of the current
 * weights), GPT2_ERR_CUDA. */
GPT2_API int gpt2_decode_step(gpt2_model* m, const int32_t* tokens, int32_t pos, float temperature,
                              const float* uniforms, int32_t* next_tokens);
/* The scores [B, Vp] (as fp32; pad columns 0) of the last decode step.
 * Synchronises.  GPT2_ERR_STATE before the first decode step. */
GPT2_API int gpt2_copy_decode_logits_out(gpt2_model* m, float* host_dst);

/* ---------------------------------------------------------------- FP8 matmuls
 * Lower precision for the matmuls (QbitAI's account of llm.c: precision can
 * go from fp32 to fp16 or lower).  E4M3 codes (OCP 8-bit float: 1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, largest finite 448, no
 * infinity) with one scale per tensor.  These entry points need no
 * gpt2_model; all pointers are device pointers owned by the caller, all work
 * is enqueued on cuda_stream (NULL = legacy stream) and nothing is
 * allocated.
 *
 * gpt2_fp8_quantize: x [n] (fp32, or bf16 if x_is_bf16) -> q [n] codes and
 *   scale[0] = s = 448 / max|x| (1 if x is all zeros; NaN entries are left
 *   out of the maximum), q[i] = E4M3(x[i] * s) with the product in fp32,
 *   rounded to nearest (ties to even), saturating at +-448 (NaN -> 0x7F).
 *   scale points to 2 floats; scale[1] is scratch.  x and q 16-byte aligned.
 * gpt2_fp8_matmul: out[m, n] = (sum_k E(a[m, k]) E(b[n, k])) /
 *   (scale_a[0] * scale_b[0]) + bias[n] (bias may be NULL; 16-byte aligned), with E the code's
 *   value; a [M, K] and b [N, K] row-major codes with row strides lda, ldb
 *   bytes (multiples of 16, >= K); out [M, N] fp32 (or bf16 if out_is_bf16)
 *   with row stride ldo elements (16-byte rows); the products accumulate in
 *   fp32 on the tensor cores (tcgen05 kind::f8f6f4).  scale_a / scale_b are
 *   the scale[0] words of the two quantisations (device).
 * gpt2_fp8_check: synchronises cuda_stream and reports a bounded device
 *   wait of these entry points that expired (GPT2_ERR_TIMEOUT), then clears it.
 * Errors: GPT2_ERR_ARG (NULL pointer, size below 1, misaligned pointer or
 * stride), GPT2_ERR_CUDA (a launch failed); gpt2_last_error(NULL) has the text. */
GPT2_API int gpt2_fp8_quantize(const void* x, int32_t x_is_bf16, int64_t n, uint8_t* q, float* scale,
                               void* cuda_stream);
GPT2_API int gpt2_fp8_matmul(const uint8_t* a, int64_t lda, const float* scale_a, const uint8_t* b,
                             int64_t ldb, const float* scale_b, int32_t M, int32_t N, int32_t K,
                             const float* bias, void* out, int64_t ldo, int32_t out_is_bf16,
                             void* cuda_stream);
GPT2_API int gpt2_fp8_check(void* cuda_stream);

/* ---------------------------------------------------------------- checkpoints
 * Training state saved and resumed as one flat file: InfoQ's account of
 * llm.c loads its model as a checkpoint file of fp32 weights in one block;
 * femtoGPT resumes training from its saved state.  The page gives no
 * layout; this one is:
 *   64 little-endian int32 header words: [0] magic 0x43545047 ("GPTC"),
 *   [1] version 1, [2] header words (64), [3..11] max_seq_len, vocab_size,
 *   padded_vocab_size, num_layers, num_heads, channels, batch_size, seq_len,
 *   precision of the saving model, [12] the step t, [13], [14] the number of
 *   fp32 parameters (low, high 32 bits), [15] the arenas that follow (3:
 *   params, AdamW m, AdamW v); the rest 0;
 *   then each arena as n_params fp32 values, in gpt2_tensor_info's order.
 * gpt2_save_checkpoint synchronises the model's stream and writes the file
 * (step >= 0 is stored as given).  gpt2_load_checkpoint needs a file whose
 * max_seq_len, vocab_size, padded_vocab_size, num_layers, num_heads,
 * channels and parameter count match the model (batch shape and precision
 * may differ); it replaces params, m and v, refreshes the bf16 weight copy,
 * zeroes the gradients, requires a new forward before the next backward, and
 * returns the saved step in *step (may be NULL).  Errors: GPT2_ERR_ARG (NULL
 * model or path, step < 0, a header that does not match), GPT2_ERR_IO
 * (open / read / write failure, short file), GPT2_ERR_CUDA; a header or
 * length check that fails leaves the model unchanged. */
GPT2_API int gpt2_save_checkpoint(gpt2_model* m, const char* path, int32_t step);
GPT2_API int gpt2_load_checkpoint(gpt2_model* m, const char* path, int32_t* step);

/* ---------------------------------------------------------------- token files
 * InfoQ's account of llm.c: the data-preparation scripts write each split
 * as a .bin file holding the raw bytes of int32 GPT-2 token ids.  A
 * gpt2_tokens reads such a file into host memory once and serves
 * next-token batches from a cursor: gpt2_tokens_next_batch copies
 * tokens[i] = s[p + i] and targets[i] = s[p + i + 1] for i < B*T (row-major
 * [B, T] host buffers owned by the caller) and advances p by B*T; a batch
 * that would read past the end starts over at p = 0.  The ids are not
 * range-checked here (gpt2_forward reports ids outside [0, V) as
 * GPT2_ERR_TOKEN).  Errors (message in gpt2_last_error(NULL)):
 * GPT2_ERR_ARG (NULL arguments, B or T < 1, a file whose size is not a
 * multiple of 4, or fewer than B*T+1 tokens), GPT2_ERR_IO (cannot read the
 * file), GPT2_ERR_OOM. */
typedef struct gpt2_tokens gpt2_tokens;
GPT2_API int gpt2_tokens_open(const char* path, gpt2_tokens** out);
GPT2_API int gpt2_tokens_count(const gpt2_tokens* d, int64_t* n);
GPT2_API int gpt2_tokens_next_batch(gpt2_tokens* d, int32_t B, int32_t T, int32_t* tokens,
                                    int32_t* targets);
GPT2_API int gpt2_tokens_reset(gpt2_tokens* d);
GPT2_API void gpt2_tokens_close(gpt2_tokens* d); /* NULL-safe */

/* Kernel timing with CUDA events recorded on the model's stream around
 * every launch of the selected kernel classes (bit i of class_mask selects
 * class i; 0 turns timing off).  Each class also accumulates the
 * algorithmic work of its launches: FLOPs of the matmuls / attention
 * contractions (2*M*N*K; causal attention counts only the unmasked half) or
 * the minimum bytes a memory-bound kernel must move (each input read once,
 * each output written once).  gpt2_profile_read synchronises and returns,
 * for class cls: its name, the unit of `work` ("flop" or "byte"), the
 * number of launches, their summed duration in milliseconds and their
 * summed work, since the last reset.  Names and units are static strings. */
GPT2_API int gpt2_profile_num_classes(int32_t* n);
GPT2_API int gpt2_profile_enable(gpt2_model* m, uint32_t class_mask);
GPT2_API int gpt2_profile_reset(gpt2_model* m);
GPT2_API int gpt2_profile_read(gpt2_model* m, int32_t cls, const char** name,
                               const char** unit, int64_t* launches,
                               double* total_ms, double* work);

/* Number of kernel launches the library made since the model was built
 * (a plain host-side counter). */
GPT2_API int gpt2_launch_count(const gpt2_model* m, int64_t* n);

/* Text of the last error on this model (or of the last failed gpt2_build
 * or model-less call when m is NULL).  Static or model-owned storage;
 * never NULL. */
GPT2_API const char* gpt2_last_error(const gpt2_model* m);

/* LayerNorm backward that allocates no device memory.  The pages have no
 * counterpart: this entry point exists for callers of this library that
 * cannot call cudaMalloc -- code whose device memory is owned by another
 * allocator (a framework's caching allocator, a fixed pool) that must not be
 * bypassed, and latency-critical loops where a cudaMalloc/cudaFree would
 * synchronise the device.  It needs no gpt2_model.
 *
 * Computes, for N rows of width C (row-major fp32, device pointers):
 *   xhat = (inp - mean) * rstd,  g = dout * weight,
 *   dinp[i]     += rstd[i] * (g - mean_row(g) - xhat * mean_row(g * xhat))
 *   dweight     += sum over rows of dout * xhat
 *   dbias       += sum over rows of dout
 *   dinp_colsum += sum over rows of the updated dinp   (skipped if NULL)
 * (the same arithmetic as the LayerNorm backward inside gpt2_backward).
 *   dinp [N, C], dweight [C], dbias [C], dinp_colsum [C] or NULL: outputs,
 *       accumulated into (the caller zeroes them for plain values);
 *   dout, inp [N, C], weight [C], mean, rstd [N]: inputs, read only;
 *   cuda_stream: the cudaStream_t to enqueue on (NULL = legacy stream).
 * Alignment: dinp, dweight, dbias, dinp_colsum, dout, inp and weight must
 * start on 16-byte boundaries (rows move by bulk copies, columns in 16-byte
 * vectors), mean and rstd on 4-byte ones; otherwise GPT2_ERR_ARG.
 * Ordering: the call's first kernel starts only after all work enqueued
 * before it on cuda_stream has finished (no programmatic overlap).
 * Scratch: the partial sums, at most ceil(N/64) * 3 * C floats, live in one
 * file-scope __device__ array of 2^21 floats (8 MiB) that every GPU which
 * loads the library holds until the process exits.  Larger sizes are
 * rejected with GPT2_ERR_ARG (N * C must stay below about 44.7 million);
 * also GPT2_ERR_ARG for a NULL input/output or C outside [4, 1024] or
 * C % 4 != 0, GPT2_ERR_CUDA if a launch fails; gpt2_last_error(NULL) has
 * the text.  Every call on a device shares the array and leaves the last
 * call's partials in it; each call writes every partial it reads, so nothing
 * needs clearing, but calls that overlap on the GPU (different streams, or
 * other threads) race on the array.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  Asynchronous;
 * calls no cudaMalloc, cudaFree or other allocating routine.  A bounded
 * device wait that expires inside the call (its outputs are then incomplete)
 * sets a per-device error word that gpt2_noalloc_check reports. */
GPT2_API int gpt2_layernorm_backward_noalloc(float* dinp, float* dweight, float* dbias,
                                             float* dinp_colsum, const float* dout,
                                             const float* inp, const float* weight,
                                             const float* mean, const float* rstd, int32_t N,
                                             int32_t C, void* cuda_stream);

/* gpt2_noalloc_check: synchronises cuda_stream, then reads and clears the
 * current device's error word of gpt2_layernorm_backward_noalloc.  Returns
 * GPT2_ERR_TIMEOUT if a bounded wait of an earlier call expired (that call's
 * outputs are incomplete), GPT2_ERR_CUDA if the stream reports a CUDA error,
 * else GPT2_OK.  Allocates nothing. */
GPT2_API int gpt2_noalloc_check(void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_H */
