"""The C-ABI library loads on a CPU-only host, exports every symbol the
public headers declare, and rejects bad arguments before touching a GPU."""
import ctypes
import glob
import os
import re

import pytest

import transformer_lm_step_gpt_b300 as tl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"GPT2_API\s+[\w\s\*]+?\b(gpt2_\w+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = tl.load_library()
    names = declared_symbols()
    assert len(names) >= 19
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_symbol():
    src = open(os.path.join(ROOT, "transformer_lm_step_gpt_b300", "__init__.py")).read()
    for n in declared_symbols():
        assert '"%s"' % n in src, n


@pytest.mark.parametrize("bad", [
    dict(C=60, NH=4),            # C % 8 != 0
    dict(C=64, NH=3),            # C % NH != 0
    dict(C=64, NH=1),            # head size 64 ok... but Vp < V below
    dict(T=40, maxT=32),         # T > maxT
    dict(V=300, Vp=256),         # V > Vp
    dict(Vp=260, V=256),         # Vp % 8 != 0
    dict(L=0),                   # no layers
    dict(B=64, T=1024, maxT=1024),  # B*T > 32768
    dict(C=1280, NH=20),         # C > 1024
    dict(B=0),                   # no sequences
    dict(T=0),                   # empty sequences
    dict(maxT=8192, T=32),       # maxT > 4096
    dict(C=96, NH=1),            # head size 96: not 16, 32, 64 or 128
    dict(C=64, NH=8),            # head size 8
    dict(V=0),                   # empty vocabulary
    dict(V=131072, Vp=131072, B=32, T=1024, maxT=1024),  # Vp*B*T = 2^32: the encoder's sort key would not fit
])
def test_build_rejects_bad_config_without_gpu(bad):
    cfg = dict(L=2, C=64, NH=4, V=256, Vp=256, maxT=32, B=4, T=32)
    cfg.update(bad)
    if bad == dict(C=64, NH=1):
        cfg.update(V=300, Vp=256)
    with pytest.raises(tl.GPT2Error) as e:
        tl.Model(cfg["L"], cfg["C"], cfg["NH"], cfg["V"], cfg["Vp"], cfg["maxT"], cfg["B"], cfg["T"],
                 precision="bf16")
    assert e.value.code == -1  # GPT2_ERR_ARG


def test_null_model_calls_return_arg_error():
    lib = tl.load_library()
    assert lib.gpt2_zero_grad(None) == -1
    assert lib.gpt2_backward(None) == -1
    assert lib.gpt2_adamw_step(None, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1) == -1
    assert lib.gpt2_forward(None, None, None, None) == -1
    lib.gpt2_free(None)  # NULL is allowed
    assert lib.gpt2_last_error(None)  # never NULL


def test_generation_and_fp8_entry_points_check_arguments_without_gpu():
    lib = tl.load_library()
    # generation: a NULL model
    assert lib.gpt2_decode_step(None, None, 0, 1.0, None, None) == -1
    assert lib.gpt2_copy_decode_logits_out(None, None) == -1
    # FP8: NULL pointers, sizes below 1, misaligned pointers and strides are
    # refused before any device work
    assert lib.gpt2_fp8_quantize(None, 0, 16, None, None, None) == -1
    assert b"NULL" in lib.gpt2_last_error(None)
    buf = ctypes.create_string_buffer(4096)
    p = (ctypes.addressof(buf) + 255) & ~255   # an aligned host address, never dereferenced here
    assert lib.gpt2_fp8_quantize(p, 0, 0, p, p, None) == -1          # n < 1
    assert lib.gpt2_fp8_quantize(p + 4, 0, 16, p, p, None) == -1     # x not 16-byte aligned
    args = dict(lda=64, ldb=64, M=8, N=8, K=64, ldo=8)

    def mm(**kw):
        a = dict(args, **kw)
        return lib.gpt2_fp8_matmul(p, a["lda"], p, p, a["ldb"], p, a["M"], a["N"], a["K"], None, p, a["ldo"], 0,
                                   None)
    assert mm(lda=40) == -1      # not a multiple of 16
    assert mm(ldb=32) == -1      # smaller than K
    assert mm(ldo=6) == -1       # ldo < N
    assert mm(M=0) == -1
    assert lib.gpt2_fp8_matmul(p, 64, p, p, 64, p, 8, 8, 64, p + 4, p, 8, 0, None) == -1   # bias misaligned
    assert b"aligned" in lib.gpt2_last_error(None)


def test_named_copies_reject_a_null_model():
    lib = tl.load_library()
    for fn in (lib.gpt2_copy_params_out, lib.gpt2_copy_grads_out, lib.gpt2_copy_m_out, lib.gpt2_copy_v_out,
               lib.gpt2_copy_params_in):
        assert fn(None, None) == -1
    out = ctypes.c_void_p()
    assert lib.gpt2_loss_device_ptr(None, ctypes.byref(out)) == -1


def test_expire_a_wait_rejects_a_null_model():
    assert tl.load_library().gpt2_expire_a_wait(None) == -1


def test_the_logits_limit_is_exact():
    # Vp*B*T = 131064*32768 < 2^32 passes the argument checks (without a GPU
    # the build then fails at the device, never with GPT2_ERR_ARG)
    try:
        m = tl.Model(1, 1024, 16, 131064, 131064, 1024, 32, 1024, precision="bf16")
        m.close()
    except tl.GPT2Error as e:
        assert e.code != -1, str(e)


def test_noalloc_layernorm_backward_checks_arguments_without_gpu():
    # gpt2_layernorm_backward_noalloc refuses NULL buffers, sizes beyond its
    # static scratch and misaligned addresses before any device work (the
    # addresses below are never dereferenced)
    lib = tl.load_library()
    buf = ctypes.create_string_buffer(4096)
    p = (ctypes.addressof(buf) + 255) & ~255
    ptrs = [p] * 9

    def call(ptrs, N=150, C=64):
        return lib.gpt2_layernorm_backward_noalloc(*[ctypes.c_void_p(x) for x in ptrs], N, C, None)
    assert call([p, p, p, p, None, p, p, p, p]) == -1
    assert b"NULL" in lib.gpt2_last_error(None)
    assert call(ptrs, N=1 << 20, C=1024) == -1
    assert b"static scratch" in lib.gpt2_last_error(None)
    assert call(ptrs, C=62) == -1          # C % 4 != 0
    for i in range(7):  # dinp, dweight, dbias, dinp_colsum, dout, inp, weight: 16-byte
        bad = list(ptrs)
        bad[i] = p + 4
        assert call(bad) == -1, i
        assert b"aligned" in lib.gpt2_last_error(None)
    for i in (7, 8):    # mean, rstd: 4-byte
        bad = list(ptrs)
        bad[i] = p + 2
        assert call(bad) == -1, i


def test_build_rejects_a_vocabulary_beyond_18_bit_token_ids():
    # the encoder backward sorts positions by token id in two 9-bit radix
    # passes, so Vp is capped at 2^18
    with pytest.raises(tl.GPT2Error) as e:
        tl.Model(1, 64, 1, 262152, 262152, 8, 1, 8, precision="bf16")
    assert e.value.code == -1
