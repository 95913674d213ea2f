"""B300-native GPT-2 training step: Python binding of libgpt2.so.

A thin ctypes layer over the C ABI in ``include/gpt2.h``: it marshals
arguments and raises :class:`GPT2Error` on a non-zero status.  Every step of
the computation runs in the library's CUDA kernels; there is no Python or CPU
fallback -- if ``libgpt2.so`` is missing or fails to load, using the binding
raises immediately.  PyTorch is used only for device memory of the token
buffers and for streams.

    from transformer_lm_step_gpt_b300 import Model
    m = Model(L=12, C=768, NH=12, V=50257, Vp=50304, maxT=1024, B=16, T=1024,
              precision="bf16", seed=1337)
    loss = m.forward(tokens, targets)        # int32 CUDA tensors [B, T]
    m.zero_grad(); m.backward(); m.adamw_step(6e-4, 0.9, 0.999, 1e-8, 0.1, t=1)
"""
import ctypes
import os

import numpy as np

__all__ = ["Model", "GPT2Error", "TokenFile", "library_path", "load_library", "layernorm_backward_noalloc", "noalloc_check",
           "fp8_quantize", "fp8_matmul", "fp8_check",
           "PARAMS", "GRADS", "ADAM_M", "ADAM_V"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgpt2.so")
_lib = None

PARAMS, GRADS, ADAM_M, ADAM_V = 0, 1, 2, 3
FP32, BF16 = 0, 1

ERRORS = {0: "OK", -1: "GPT2_ERR_ARG", -2: "GPT2_ERR_OOM", -3: "GPT2_ERR_CUDA", -4: "GPT2_ERR_STATE",
          -5: "GPT2_ERR_TOKEN", -6: "GPT2_ERR_TIMEOUT", -7: "GPT2_ERR_NONFINITE", -8: "GPT2_ERR_IO"}


class GPT2Error(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s (%d): %s" % (ERRORS.get(code, "?"), code, msg))
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("max_seq_len", ctypes.c_int32), ("vocab_size", ctypes.c_int32),
                ("padded_vocab_size", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("channels", ctypes.c_int32),
                ("batch_size", ctypes.c_int32), ("seq_len", ctypes.c_int32),
                ("precision", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libgpt2.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libgpt2.so is not built; run `python -m transformer_lm_step_gpt_b300.build` "
                           "(there is no CPU fallback)")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sig = {
        "gpt2_build": ([ctypes.POINTER(Config), ctypes.c_uint64, ctypes.POINTER(vp)], ctypes.c_int),
        "gpt2_free": ([vp], None),
        "gpt2_set_stream": ([vp, vp], ctypes.c_int),
        "gpt2_forward": ([vp, vp, vp, vp], ctypes.c_int),
        "gpt2_forward_host": ([vp, vp, vp, vp], ctypes.c_int),
        "gpt2_zero_grad": ([vp], ctypes.c_int),
        "gpt2_backward": ([vp], ctypes.c_int),
        "gpt2_adamw_step": ([vp, f32, f32, f32, f32, f32, i32], ctypes.c_int),
        "gpt2_synchronize": ([vp], ctypes.c_int),
        "gpt2_expire_a_wait": ([vp], ctypes.c_int),
        "gpt2_get_config": ([vp, ctypes.POINTER(Config)], ctypes.c_int),
        "gpt2_num_params": ([vp, ctypes.POINTER(i64)], ctypes.c_int),
        "gpt2_num_tensors": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
        "gpt2_tensor_info": ([vp, i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i64),
                              ctypes.POINTER(i64)], ctypes.c_int),
        "gpt2_copy_out": ([vp, i32, vp], ctypes.c_int),
        "gpt2_copy_in": ([vp, i32, vp], ctypes.c_int),
        "gpt2_copy_params_out": ([vp, vp], ctypes.c_int),
        "gpt2_copy_grads_out": ([vp, vp], ctypes.c_int),
        "gpt2_copy_m_out": ([vp, vp], ctypes.c_int),
        "gpt2_copy_v_out": ([vp, vp], ctypes.c_int),
        "gpt2_copy_params_in": ([vp, vp], ctypes.c_int),
        "gpt2_loss_device_ptr": ([vp, ctypes.POINTER(vp)], ctypes.c_int),
        "gpt2_copy_losses_out": ([vp, vp], ctypes.c_int),
        "gpt2_copy_logits_out": ([vp, vp], ctypes.c_int),
        "gpt2_copy_residual_out": ([vp, i32, vp], ctypes.c_int),
        "gpt2_read_loss": ([vp, ctypes.POINTER(f32)], ctypes.c_int),
        "gpt2_profile_num_classes": ([ctypes.POINTER(i32)], ctypes.c_int),
        "gpt2_profile_enable": ([vp, ctypes.c_uint32], ctypes.c_int),
        "gpt2_profile_reset": ([vp], ctypes.c_int),
        "gpt2_profile_read": ([vp, i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_char_p),
                               ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_double)], ctypes.c_int),
        "gpt2_launch_count": ([vp, ctypes.POINTER(i64)], ctypes.c_int),
        "gpt2_last_error": ([vp], ctypes.c_char_p),
        "gpt2_layernorm_backward_noalloc": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp], ctypes.c_int),
        "gpt2_noalloc_check": ([vp], ctypes.c_int),
        "gpt2_save_checkpoint": ([vp, ctypes.c_char_p, i32], ctypes.c_int),
        "gpt2_load_checkpoint": ([vp, ctypes.c_char_p, ctypes.POINTER(i32)], ctypes.c_int),
        "gpt2_tokens_open": ([ctypes.c_char_p, ctypes.POINTER(vp)], ctypes.c_int),
        "gpt2_tokens_count": ([vp, ctypes.POINTER(i64)], ctypes.c_int),
        "gpt2_tokens_next_batch": ([vp, i32, i32, vp, vp], ctypes.c_int),
        "gpt2_tokens_reset": ([vp], ctypes.c_int),
        "gpt2_tokens_close": ([vp], None),
        "gpt2_decode_step": ([vp, vp, i32, f32, vp, vp], ctypes.c_int),
        "gpt2_fp8_quantize": ([vp, i32, i64, vp, vp, vp], ctypes.c_int),
        "gpt2_fp8_matmul": ([vp, i64, vp, vp, i64, vp, i32, i32, i32, vp, vp, i64, i32, vp], ctypes.c_int),
        "gpt2_fp8_check": ([vp], ctypes.c_int),
        "gpt2_copy_decode_logits_out": ([vp, vp], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _buf(x, n, dtype, where, name):
    """Address of a buffer in which the library reads or writes n elements of
    dtype ("int32", "float32", ...); where is "cuda" (device memory) or
    "host".  A torch tensor or numpy array is checked first (its device, its
    dtype, contiguity, at least n elements), so that a wrong buffer raises
    here instead of being read or written past its end; a raw int address is
    passed on unchecked; None is NULL."""
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):  # a torch tensor
        if bool(x.is_cuda) != (where == "cuda"):
            raise ValueError("%s: need a %s tensor" % (name, "CUDA" if where == "cuda" else "host (CPU)"))
        dt, contiguous, numel, addr = str(x.dtype).replace("torch.", ""), x.is_contiguous(), x.numel(), x.data_ptr()
    elif isinstance(x, np.ndarray):
        if where == "cuda":
            raise ValueError("%s: need a CUDA tensor, not a numpy array" % name)
        dt, contiguous, numel, addr = str(x.dtype), bool(x.flags["C_CONTIGUOUS"]), x.size, x.ctypes.data
    else:
        raise TypeError("%s: unsupported buffer type %s" % (name, type(x).__name__))
    if dt != dtype:
        raise TypeError("%s: dtype %s, need %s" % (name, dt, dtype))
    if not contiguous:
        raise ValueError("%s: must be contiguous" % name)
    if numel < n:
        raise ValueError("%s: %d elements, need %d" % (name, numel, n))
    return addr


class Model:
    """One GPT-2 model with all of its device memory (see include/gpt2.h)."""

    def __init__(self, L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=1337, stream=None):
        self._lib = load_library()
        self.cfg = Config(maxT, V, Vp, L, NH, C, B, T, BF16 if precision == "bf16" else FP32)
        self.L, self.C, self.NH, self.V, self.Vp, self.maxT, self.B, self.T = L, C, NH, V, Vp, maxT, B, T
        self.precision = precision
        h = ctypes.c_void_p()
        rc = self._lib.gpt2_build(ctypes.byref(self.cfg), ctypes.c_uint64(seed), ctypes.byref(h))
        if rc != 0:
            raise GPT2Error(rc, self._lib.gpt2_last_error(None).decode())
        self._h = h
        if stream is not None:
            self.set_stream(stream)

    # -- lifetime --------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            self._lib.gpt2_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != 0:
            raise GPT2Error(rc, self._lib.gpt2_last_error(self._h).decode())

    # -- the step ----------------------------------------------------------
    def set_stream(self, stream):
        """stream: a torch.cuda.Stream, a raw cudaStream_t int, or None."""
        s = getattr(stream, "cuda_stream", stream)
        self._check(self._lib.gpt2_set_stream(self._h, s))

    def forward(self, tokens, targets=None, sync=True):
        """tokens/targets: int32 device tensors [B, T].  Returns the mean loss
        (a float) when sync and targets are given, else None."""
        M = self.B * self.T
        tok = _buf(tokens, M, "int32", "cuda", "tokens")
        tgt = _buf(targets, M, "int32", "cuda", "targets")
        loss = ctypes.c_float(float("nan"))
        self._check(self._lib.gpt2_forward(self._h, tok, tgt, ctypes.byref(loss) if sync else None))
        return loss.value if (sync and targets is not None) else None

    def forward_host(self, tokens, targets=None, sync=True):
        """As forward, with host (ideally pinned) int32 buffers."""
        M = self.B * self.T
        tok = _buf(tokens, M, "int32", "host", "tokens")
        tgt = _buf(targets, M, "int32", "host", "targets")
        loss = ctypes.c_float(float("nan"))
        self._check(self._lib.gpt2_forward_host(self._h, tok, tgt, ctypes.byref(loss) if sync else None))
        return loss.value if (sync and targets is not None) else None

    def zero_grad(self):
        self._check(self._lib.gpt2_zero_grad(self._h))

    def backward(self):
        self._check(self._lib.gpt2_backward(self._h))

    def adamw_step(self, lr, beta1, beta2, eps, weight_decay, t):
        self._check(self._lib.gpt2_adamw_step(self._h, lr, beta1, beta2, eps, weight_decay, int(t)))

    def expire_a_wait(self):
        """Enqueue a kernel whose bounded wait runs out (see gpt2_expire_a_wait):
        the next synchronising call raises GPT2_ERR_TIMEOUT."""
        self._check(self._lib.gpt2_expire_a_wait(self._h))

    def synchronize(self):
        self._check(self._lib.gpt2_synchronize(self._h))

    # -- inspection -------------------------------------------------------
    @property
    def num_params(self) -> int:
        n = ctypes.c_int64()
        self._check(self._lib.gpt2_num_params(self._h, ctypes.byref(n)))
        return n.value

    def tensor_table(self):
        n = ctypes.c_int32()
        self._check(self._lib.gpt2_num_tensors(self._h, ctypes.byref(n)))
        out = []
        for i in range(n.value):
            name, off, cnt = ctypes.c_char_p(), ctypes.c_int64(), ctypes.c_int64()
            self._check(self._lib.gpt2_tensor_info(self._h, i, ctypes.byref(name), ctypes.byref(off),
                                                   ctypes.byref(cnt)))
            out.append((name.value.decode(), off.value, cnt.value))
        return out

    def copy_out(self, arena=PARAMS) -> np.ndarray:
        a = np.empty(self.num_params, np.float32)
        self._check(self._lib.gpt2_copy_out(self._h, arena, a.ctypes.data))
        return a

    def copy_in(self, arr, arena=PARAMS):
        a = np.ascontiguousarray(arr, dtype=np.float32)
        if a.size != self.num_params:
            raise ValueError("copy_in: %d values, the arena holds %d" % (a.size, self.num_params))
        self._check(self._lib.gpt2_copy_in(self._h, arena, a.ctypes.data))

    def losses(self) -> np.ndarray:
        a = np.empty(self.B * self.T, np.float32)
        self._check(self._lib.gpt2_copy_losses_out(self._h, a.ctypes.data))
        return a

    def logits(self) -> np.ndarray:
        a = np.empty((self.B * self.T, self.Vp), np.float32)
        self._check(self._lib.gpt2_copy_logits_out(self._h, a.ctypes.data))
        return a

    def residual(self, layer) -> np.ndarray:
        """fp32 residual stream [B*T, C] entering block `layer` (0 = encoder output)."""
        a = np.empty((self.B * self.T, self.C), np.float32)
        self._check(self._lib.gpt2_copy_residual_out(self._h, int(layer), a.ctypes.data))
        return a

    def loss_device_ptr(self) -> int:
        """Device address of the fp32 mean loss of the last forward with targets."""
        p = ctypes.c_void_p()
        self._check(self._lib.gpt2_loss_device_ptr(self._h, ctypes.byref(p)))
        return p.value

    def read_loss(self) -> float:
        """Mean loss of the last forward with targets (synchronises)."""
        x = ctypes.c_float()
        self._check(self._lib.gpt2_read_loss(self._h, ctypes.byref(x)))
        return x.value

    def profile_enable(self, classes="all"):
        """Time the named kernel classes with CUDA events (None/[] = off)."""
        n = ctypes.c_int32()
        self._check(self._lib.gpt2_profile_num_classes(ctypes.byref(n)))
        mask = 0
        if classes == "all":
            mask = (1 << n.value) - 1
        elif classes:
            names = [r["name"] for r in self.profile_read()]
            for c in classes:
                mask |= 1 << names.index(c)
        self._check(self._lib.gpt2_profile_enable(self._h, mask))

    def profile_reset(self):
        self._check(self._lib.gpt2_profile_reset(self._h))

    def profile_read(self):
        """[{name, unit, launches, ms, work}] per kernel class (synchronises)."""
        n = ctypes.c_int32()
        self._check(self._lib.gpt2_profile_num_classes(ctypes.byref(n)))
        out = []
        for i in range(n.value):
            name, unit = ctypes.c_char_p(), ctypes.c_char_p()
            cnt, ms, work = ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
            self._check(self._lib.gpt2_profile_read(self._h, i, ctypes.byref(name), ctypes.byref(unit),
                                                    ctypes.byref(cnt), ctypes.byref(ms), ctypes.byref(work)))
            out.append(dict(name=name.value.decode(), unit=unit.value.decode(), launches=cnt.value,
                            ms=ms.value, work=work.value))
        return out

    @property
    def launch_count(self) -> int:
        n = ctypes.c_int64()
        self._check(self._lib.gpt2_launch_count(self._h, ctypes.byref(n)))
        return n.value

    # -- generation ----------------------------------------------------------
    def decode_step(self, tokens, pos, temperature, uniforms, out=None):
        """One position of every sequence with the key/value cache (see
        gpt2_decode_step): tokens (int32 [B]) at position pos in, the drawn
        next tokens (int32 [B]) out; uniforms: float32 [B] in [0, 1).  All
        three are CUDA tensors used in the model's stream order."""
        if out is None:
            import torch
            dev = tokens.device if hasattr(tokens, "device") else torch.device("cuda", torch.cuda.current_device())
            out = torch.empty(self.B, dtype=torch.int32, device=dev)
        tok = _buf(tokens, self.B, "int32", "cuda", "tokens")
        u = _buf(uniforms, self.B, "float32", "cuda", "uniforms")
        nxt = _buf(out, self.B, "int32", "cuda", "out")
        self._check(self._lib.gpt2_decode_step(self._h, tok, int(pos), float(temperature), u, nxt))
        return out

    def decode_logits(self) -> np.ndarray:
        """Scores [B, Vp] of the last decode step (synchronises)."""
        a = np.empty((self.B, self.Vp), np.float32)
        self._check(self._lib.gpt2_copy_decode_logits_out(self._h, a.ctypes.data))
        return a

    def generate(self, prompt, n_new, temperature=1.0, seed=0, uniforms=None):
        """prompt: int32 [B, T0] host ids (1 <= T0 <= T).  A forward over the
        prompts (padded to T) fills the cache; then n_new decode steps at
        positions T0-1 .. T0-2+n_new each draw one token, new token i of
        sequence b with uniforms[i, b] (default: numpy's generator seeded with
        `seed`).  Returns int32 [B, T0 + n_new]: prompt, then the new tokens."""
        import torch
        prompt = np.ascontiguousarray(prompt, np.int32).reshape(self.B, -1)
        T0 = prompt.shape[1]
        if not (1 <= T0 <= self.T) or n_new < 0 or T0 - 1 + n_new > self.T:
            raise ValueError("need 1 <= T0 <= T and T0 - 1 + n_new <= T")
        if uniforms is None:
            uniforms = np.random.default_rng(seed).random((n_new, self.B))
        u = np.ascontiguousarray(uniforms, np.float32).reshape(n_new, self.B)
        dev = torch.device("cuda", torch.cuda.current_device())
        padded = np.zeros((self.B, self.T), np.int32)
        padded[:, :T0] = prompt
        tok_d = torch.from_numpy(padded).to(dev)
        seq_d = torch.empty((n_new + 1, self.B), dtype=torch.int32, device=dev)
        seq_d[0] = torch.from_numpy(np.ascontiguousarray(prompt[:, T0 - 1])).to(dev)
        u_d = torch.from_numpy(u).to(dev)
        torch.cuda.synchronize(dev)  # inputs in place before the model's stream reads them
        self.forward(tok_d, None, sync=False)
        for i in range(n_new):
            self.decode_step(seq_d[i], T0 - 1 + i, temperature, u_d[i], out=seq_d[i + 1])
        self.synchronize()
        new = seq_d[1:].cpu().numpy().T
        return np.concatenate([prompt, new], axis=1).astype(np.int32)

    # -- checkpoints ---------------------------------------------------------
    def save_checkpoint(self, path, step=0):
        """Write params, AdamW m and v and `step` to one flat file."""
        self._check(self._lib.gpt2_save_checkpoint(self._h, os.fsencode(path), int(step)))

    def load_checkpoint(self, path) -> int:
        """Replace params, m and v from a checkpoint of this model's shape;
        returns the saved step."""
        t = ctypes.c_int32()
        self._check(self._lib.gpt2_load_checkpoint(self._h, os.fsencode(path), ctypes.byref(t)))
        return t.value


class TokenFile:
    """A raw int32 token file (.bin) served as next-token batches:
    next_batch(B, T) -> (tokens, targets), int32 arrays [B, T] with
    targets[i] = tokens[i + 1] along the file, the cursor advancing by B*T
    and starting over when a batch would run past the end."""

    def __init__(self, path):
        self._lib = load_library()
        h = ctypes.c_void_p()
        rc = self._lib.gpt2_tokens_open(os.fsencode(path), ctypes.byref(h))
        if rc != 0:
            raise GPT2Error(rc, self._lib.gpt2_last_error(None).decode())
        self._h = h

    def __len__(self):
        n = ctypes.c_int64()
        self._check(self._lib.gpt2_tokens_count(self._h, ctypes.byref(n)))
        return n.value

    def _check(self, rc):
        if rc != 0:
            raise GPT2Error(rc, self._lib.gpt2_last_error(None).decode())

    def next_batch(self, B, T, tokens=None, targets=None):
        """Fill (and return) host int32 buffers of B*T elements; pinned
        torch tensors or numpy arrays may be passed in."""
        if tokens is None:
            tokens = np.empty((B, T), np.int32)
        if targets is None:
            targets = np.empty((B, T), np.int32)
        n = int(B) * int(T)
        self._check(self._lib.gpt2_tokens_next_batch(self._h, int(B), int(T), _buf(tokens, n, "int32", "host", "tokens"),
                                                     _buf(targets, n, "int32", "host", "targets")))
        return tokens, targets

    def reset(self):
        self._check(self._lib.gpt2_tokens_reset(self._h))

    def close(self):
        if getattr(self, "_h", None):
            self._lib.gpt2_tokens_close(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def layernorm_backward_noalloc(dinp, dweight, dbias, dinp_colsum, dout, inp, weight, mean, rstd,
                               N, C, stream=None):
    """gpt2_layernorm_backward_noalloc on device buffers (torch tensors or
    raw pointers); outputs are accumulated into.  Allocates nothing."""
    L = load_library()
    s = getattr(stream, "cuda_stream", stream)
    N, C = int(N), int(C)
    f = lambda x, n, name: _buf(x, n, "float32", "cuda", name)  # noqa: E731
    rc = L.gpt2_layernorm_backward_noalloc(f(dinp, N * C, "dinp"), f(dweight, C, "dweight"), f(dbias, C, "dbias"),
                                           f(dinp_colsum, C, "dinp_colsum"), f(dout, N * C, "dout"),
                                           f(inp, N * C, "inp"), f(weight, C, "weight"), f(mean, N, "mean"),
                                           f(rstd, N, "rstd"), N, C, s)
    if rc != 0:
        raise GPT2Error(rc, L.gpt2_last_error(None).decode())


def noalloc_check(stream=None):
    """gpt2_noalloc_check: synchronise the stream and raise GPT2Error if a
    bounded device wait of an earlier allocation-free call expired."""
    L = load_library()
    rc = L.gpt2_noalloc_check(getattr(stream, "cuda_stream", stream))
    if rc != 0:
        raise GPT2Error(rc, L.gpt2_last_error(None).decode())


# ---- FP8 (E4M3) matmuls with per-tensor scaling ------------------------------

def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return getattr(stream, "cuda_stream", stream)


def _check_global(rc):
    if rc != 0:
        raise GPT2Error(rc, load_library().gpt2_last_error(None).decode())


def fp8_quantize(x, stream=None):
    """x: contiguous fp32 or bf16 CUDA tensor -> (q: uint8 codes like x,
    scale: float32 [2] with scale[0] = 448 / max|x|), see gpt2_fp8_quantize."""
    import torch
    if not (isinstance(x, torch.Tensor) and x.is_cuda):
        raise ValueError("x: need a CUDA tensor")
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x: dtype %s, need float32 or bfloat16" % str(x.dtype).replace("torch.", ""))
    if not x.is_contiguous():
        raise ValueError("x: must be contiguous")
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scale = torch.empty(2, dtype=torch.float32, device=x.device)
    _check_global(load_library().gpt2_fp8_quantize(x.data_ptr(), int(x.dtype == torch.bfloat16), x.numel(),
                                                   q.data_ptr(), scale.data_ptr(), _stream_ptr(stream)))
    return q, scale


def fp8_matmul(qa, scale_a, qb, scale_b, bias=None, out_dtype=None, stream=None):
    """(E(qa) E(qb)^T) / (scale_a[0] scale_b[0]) + bias: qa [M, K], qb [N, K]
    uint8 codes (row strides multiples of 16 bytes); out [M, N] fp32 or bf16."""
    import torch
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype: need float32 or bfloat16")
    for t, name in ((qa, "qa"), (qb, "qb")):
        if not (isinstance(t, torch.Tensor) and t.is_cuda):
            raise ValueError("%s: need a CUDA tensor" % name)
        if t.dtype != torch.uint8:
            raise TypeError("%s: dtype %s, need uint8 codes" % (name, str(t.dtype).replace("torch.", "")))
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("%s: need a 2-D tensor whose rows are contiguous" % name)
    M, K = qa.shape
    N = qb.shape[0]
    if qb.shape[1] != K:
        raise ValueError("qa and qb: K differs (%d, %d)" % (K, qb.shape[1]))
    sa = _buf(scale_a, 1, "float32", "cuda", "scale_a")
    sb = _buf(scale_b, 1, "float32", "cuda", "scale_b")
    bp = _buf(bias, N, "float32", "cuda", "bias")
    out = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    _check_global(load_library().gpt2_fp8_matmul(
        qa.data_ptr(), qa.stride(0), sa, qb.data_ptr(), qb.stride(0), sb, M, N, K, bp, out.data_ptr(),
        out.stride(0), int(out_dtype == torch.bfloat16), _stream_ptr(stream)))
    return out


def fp8_check(stream=None):
    """Synchronise and report an expired device wait of the FP8 entry points."""
    _check_global(load_library().gpt2_fp8_check(_stream_ptr(stream)))
