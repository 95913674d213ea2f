"""ctypes wrapper around the CPU oracle (oracle/gpt2_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this; the product package never
does.  The oracle is a plain fp32 / fp64 CPU implementation of one GPT-2
training step (forward, backward, AdamW); see the C++ file for the passages
each function follows.

Shapes are passed as ``cfg8 = (L, C, NH, V, Vp, maxT, B, T)``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_set_threads.restype = ctypes.c_int
        L.oracle_num_params.argtypes = [_i32p]
        L.oracle_num_params.restype = _i64
        L.oracle_num_activations.argtypes = [_i32p]
        L.oracle_num_activations.restype = _i64
        L.oracle_num_param_tensors.restype = ctypes.c_int
        L.oracle_param_tensor.argtypes = [_i32p, ctypes.c_int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
        L.oracle_param_tensor.restype = ctypes.c_int
        L.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.oracle_normal_at.argtypes = [ctypes.c_uint64, _i64]
        L.oracle_normal_at.restype = ctypes.c_double
        L.oracle_init_params.argtypes = [_i32p, ctypes.c_uint64, _f64p]
        L.oracle_init_params.restype = ctypes.c_int
        for suf, fp in (("f32", _f32p), ("f64", _f64p)):
            f = getattr(L, "oracle_fwdbwd_" + suf)
            f.argtypes = [_i32p, fp, _i32p, vp, vp, vp, vp]
            f.restype = ctypes.c_double
        L.oracle_residuals_f32.argtypes = [_i32p, _f32p, _i32p, _f32p]
        L.oracle_residuals_f32.restype = ctypes.c_int
        flt, dbl = ctypes.c_float, ctypes.c_double
        L.oracle_adamw_f32.argtypes = [_i64, _f32p, _f32p, _f32p, _f32p, flt, flt, flt, flt, flt, ctypes.c_int]
        L.oracle_adamw_f64.argtypes = [_i64, _f64p, _f64p, _f64p, _f64p, dbl, dbl, dbl, dbl, dbl, ctypes.c_int]
        L.oracle_encoder_forward_f64.argtypes = [_f64p, _i32p, _f64p, _f64p, _i64, _i64, _i64]
        L.oracle_encoder_backward_f64.argtypes = [_f64p, _f64p, _f64p, _i32p, _i64, _i64, _i64]
        L.oracle_layernorm_forward_f64.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _i64, _i64]
        L.oracle_layernorm_backward_f64.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _i64, _i64]
        L.oracle_matmul_forward_f64.argtypes = [_f64p, _f64p, _f64p, vp, _i64, _i64, _i64]
        L.oracle_matmul_backward_f64.argtypes = [_f64p, _f64p, vp, _f64p, _f64p, _f64p, _i64, _i64, _i64]
        L.oracle_attention_forward_f64.argtypes = [_f64p, _f64p, _f64p, _f64p, _i64, _i64, _i64, _i64]
        L.oracle_attention_backward_f64.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _i64, _i64, _i64, _i64]
        L.oracle_gelu_forward_f64.argtypes = [_f64p, _f64p, _i64]
        L.oracle_gelu_backward_f64.argtypes = [_f64p, _f64p, _f64p, _i64]
        L.oracle_crossentropy_forward_f64.argtypes = [_f64p, _f64p, _f64p, vp, _i64, _i64]
        L.oracle_crossentropy_backward_f64.argtypes = [_f64p, _f64p, _i32p, _i64, _i64, ctypes.c_double]
        L.oracle_decode_logits_f64.argtypes = [_i32p, _f64p, _i32p, _f64p]
        L.oracle_decode_logits_f64.restype = ctypes.c_int
        L.oracle_generate_f64.argtypes = [_i32p, _f64p, _i32p, _i64, _i64, ctypes.c_double, _f64p, _i32p, vp]
        L.oracle_generate_f64.restype = ctypes.c_int
        L.oracle_sample_f64.argtypes = [_f64p, _i64, ctypes.c_double, ctypes.c_double]
        L.oracle_sample_f64.restype = _i64
        _u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_fp8_quantize.argtypes = [_f32p, _i64, _u8p]
        L.oracle_fp8_quantize.restype = ctypes.c_float
        L.oracle_fp8_matmul.argtypes = [_f64p, _u8p, ctypes.c_double, _u8p, ctypes.c_double, vp, _i64, _i64, _i64]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def cfg8(L, C, NH, V, Vp, maxT, B, T):
    return np.array([L, C, NH, V, Vp, maxT, B, T], dtype=np.int32)


def set_threads(n: int = 0) -> int:
    return lib().oracle_set_threads(int(n))


def num_params(cfg) -> int:
    return int(lib().oracle_num_params(cfg))


def num_activations(cfg) -> int:
    return int(lib().oracle_num_activations(cfg))


PARAM_NAMES = ["wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"]


def param_table(cfg):
    """[(name, offset, numel)] of the parameter tensors in the 1-D array."""
    L = lib()
    out = []
    for i in range(L.oracle_num_param_tensors()):
        off, n = _i64(), _i64()
        assert L.oracle_param_tensor(cfg, i, ctypes.byref(off), ctypes.byref(n)) == 0
        out.append((PARAM_NAMES[i], off.value, n.value))
    return out


def philox4x32_10(ctr, key):
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(np.asarray(ctr, np.uint32), np.asarray(key, np.uint32), out)
    return out


def normal_at(seed: int, e: int) -> float:
    return lib().oracle_normal_at(seed, e)


def init_params(cfg, seed: int) -> np.ndarray:
    out = np.zeros(num_params(cfg), np.float64)
    assert lib().oracle_init_params(cfg, seed, out) == 0
    return out


def fwdbwd(cfg, params, tokens, targets=None, want_grads=True, want_logits=False):
    """Forward (+ backward) of the whole model.

    Returns dict(loss, losses, grads, logits); dtype follows ``params``
    (float32 -> the fp32 oracle, float64 -> the fp64 one).
    """
    params = np.ascontiguousarray(params)
    dt = params.dtype
    f = lib().oracle_fwdbwd_f32 if dt == np.float32 else lib().oracle_fwdbwd_f64
    B, T, V = int(cfg[6]), int(cfg[7]), int(cfg[3])
    tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
    tg = None if targets is None else np.ascontiguousarray(targets, np.int32).reshape(-1)
    grads = np.zeros_like(params) if (want_grads and tg is not None) else None
    losses = np.zeros(B * T, dt) if tg is not None else None
    logits = np.zeros(B * T * V, dt) if want_logits else None
    loss = f(cfg, params, tokens, _ptr(tg), _ptr(grads), _ptr(losses), _ptr(logits))
    return dict(loss=loss, losses=losses, grads=grads,
                logits=None if logits is None else logits.reshape(B * T, V))


def residuals_f32(cfg, params, tokens):
    """fp32 residual streams [(L+1), B*T, C] of a forward pass."""
    L, C, B, T = int(cfg[0]), int(cfg[1]), int(cfg[6]), int(cfg[7])
    out = np.zeros((L + 1, B * T, C), np.float32)
    assert lib().oracle_residuals_f32(cfg, np.ascontiguousarray(params, np.float32),
                                      np.ascontiguousarray(tokens, np.int32).reshape(-1), out) == 0
    return out


def adamw(params, grads, m, v, lr, b1, b2, eps, wd, t):
    """In-place AdamW update of params, m, v (float32 or float64 arrays)."""
    n = params.size
    if params.dtype == np.float32:
        lib().oracle_adamw_f32(n, params, grads, m, v, lr, b1, b2, eps, wd, int(t))
    else:
        lib().oracle_adamw_f64(n, params, grads, m, v, lr, b1, b2, eps, wd, int(t))


def step(cfg, params, m, v, tokens, targets, lr, b1, b2, eps, wd, t):
    """One training step (forward, backward, AdamW) in place; returns the
    pre-update mean loss and the gradients."""
    r = fwdbwd(cfg, params, tokens, targets, want_grads=True)
    adamw(params, r["grads"], m, v, lr, b1, b2, eps, wd, t)
    return r["loss"], r["grads"], r["losses"]


# ---- generation with a key/value cache (double) ----------------------------

def decode_logits(cfg, params, tokens):
    """Logits [B, T, V] of every position, computed one position at a time
    with the key/value cache (the incremental form of the forward)."""
    B, T, V = int(cfg[6]), int(cfg[7]), int(cfg[3])
    out = np.zeros(B * T * V)
    assert lib().oracle_decode_logits_f64(cfg, np.ascontiguousarray(params, np.float64),
                                          np.ascontiguousarray(tokens, np.int32).reshape(-1), out) == 0
    return out.reshape(B, T, V)


def generate(cfg, params, prompt, n_new, temperature, uniforms):
    """Prompt [B, T0] -> (tokens [B, T0 + n_new], logits [n_new, B, V]); new
    token i of sequence b is drawn with uniforms[i, b]."""
    B, V = int(cfg[6]), int(cfg[3])
    prompt = np.ascontiguousarray(prompt, np.int32).reshape(B, -1)
    T0 = prompt.shape[1]
    u = np.ascontiguousarray(uniforms, np.float64).reshape(-1)
    assert u.size == n_new * B
    toks = np.zeros((B, T0 + n_new), np.int32)
    logits = np.zeros(max(n_new, 1) * B * V)
    assert lib().oracle_generate_f64(cfg, np.ascontiguousarray(params, np.float64), prompt.reshape(-1),
                                     T0, n_new, float(temperature), u, toks, _ptr(logits)) == 0
    return toks, logits[:n_new * B * V].reshape(n_new, B, V)


def sample(logits, temperature, u):
    """Index drawn from one row of scores (inverse CDF of the softmax at the
    temperature; greedy for temperature <= 0)."""
    lg = np.ascontiguousarray(logits, np.float64).reshape(-1)
    return int(lib().oracle_sample_f64(lg, lg.size, float(temperature), float(u)))


# ---- FP8 (E4M3) with per-tensor scaling -------------------------------------

def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code)))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(x)))


def fp8_quantize(x):
    """(codes uint8 like x, scale s = 448 / max|x|) for a float32 array."""
    x = np.ascontiguousarray(x, np.float32)
    q = np.zeros(x.shape, np.uint8)
    s = lib().oracle_fp8_quantize(x.reshape(-1), x.size, q.reshape(-1))
    return q, float(np.float32(s))


def fp8_matmul(qa, sa, qb, sb, bias=None):
    """qa [M, K], qb [N, K] uint8 codes -> (dec(qa) dec(qb)^T) / (sa sb) + bias, float64 [M, N]."""
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    M, K = qa.shape
    N = qb.shape[0]
    out = np.zeros((M, N))
    b = None if bias is None else np.ascontiguousarray(bias, np.float64)
    lib().oracle_fp8_matmul(out, qa, float(sa), qb, float(sb), _ptr(b), M, N, K)
    return out


# ---- layer primitives (double) -------------------------------------------

def encoder_forward(tok, wte, wpe, B, T, C):
    out = np.zeros(B * T * C)
    lib().oracle_encoder_forward_f64(out, np.ascontiguousarray(tok, np.int32).reshape(-1),
                                     wte, wpe, B, T, C)
    return out


def encoder_backward(dout, tok, Vrows, B, T, C, maxT):
    dwte = np.zeros(Vrows * C)
    dwpe = np.zeros(maxT * C)
    lib().oracle_encoder_backward_f64(dwte, dwpe, dout, np.ascontiguousarray(tok, np.int32).reshape(-1), B, T, C)
    return dwte, dwpe


def layernorm_forward(x, w, b):
    N, C = x.shape
    out = np.zeros((N, C)); mean = np.zeros(N); rstd = np.zeros(N)
    lib().oracle_layernorm_forward_f64(out, mean, rstd, np.ascontiguousarray(x), w, b, N, C)
    return out, mean, rstd


def layernorm_backward(dout, x, w, mean, rstd):
    N, C = x.shape
    dx = np.zeros((N, C)); dw = np.zeros(C); db = np.zeros(C)
    lib().oracle_layernorm_backward_f64(dx, dw, db, np.ascontiguousarray(dout), np.ascontiguousarray(x),
                                        w, mean, rstd, N, C)
    return dx, dw, db


def matmul_forward(x, W, bias=None):
    N, IC = x.shape
    OC = W.shape[0]
    out = np.zeros((N, OC))
    lib().oracle_matmul_forward_f64(out, np.ascontiguousarray(x), np.ascontiguousarray(W), _ptr(bias), N, IC, OC)
    return out


def matmul_backward(dout, x, W, with_bias=True):
    N, IC = x.shape
    OC = W.shape[0]
    dx = np.zeros((N, IC)); dW = np.zeros((OC, IC)); db = np.zeros(OC) if with_bias else None
    lib().oracle_matmul_backward_f64(dx, dW, _ptr(db), np.ascontiguousarray(dout), np.ascontiguousarray(x),
                                     np.ascontiguousarray(W), N, IC, OC)
    return dx, dW, db


def attention_forward(qkv, B, T, C, NH):
    out = np.zeros((B, T, C)); pre = np.zeros((B, NH, T, T)); att = np.zeros((B, NH, T, T))
    lib().oracle_attention_forward_f64(out, pre, att, np.ascontiguousarray(qkv, np.float64), B, T, C, NH)
    return out, pre, att


def attention_backward(dout, qkv, att, B, T, C, NH):
    dqkv = np.zeros((B, T, 3 * C)); dpre = np.zeros((B, NH, T, T)); datt = np.zeros((B, NH, T, T))
    lib().oracle_attention_backward_f64(dqkv, dpre, datt, np.ascontiguousarray(dout), np.ascontiguousarray(qkv),
                                        np.ascontiguousarray(att), B, T, C, NH)
    return dqkv


def gelu_forward(x):
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros_like(x)
    lib().oracle_gelu_forward_f64(out, x, x.size)
    return out


def gelu_backward(x, dout):
    x = np.ascontiguousarray(x, np.float64)
    d = np.zeros_like(x)
    lib().oracle_gelu_backward_f64(d, x, np.ascontiguousarray(dout, np.float64), x.size)
    return d


def crossentropy_forward(logits, targets=None):
    N, V = logits.shape
    losses = np.zeros(N); probs = np.zeros((N, V))
    tg = None if targets is None else np.ascontiguousarray(targets, np.int32)
    lib().oracle_crossentropy_forward_f64(losses, probs, np.ascontiguousarray(logits), _ptr(tg), N, V)
    return losses, probs


def crossentropy_backward(probs, targets, dloss):
    N, V = probs.shape
    d = np.zeros((N, V))
    lib().oracle_crossentropy_backward_f64(d, np.ascontiguousarray(probs), np.ascontiguousarray(targets, np.int32),
                                           N, V, dloss)
    return d
