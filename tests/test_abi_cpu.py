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
