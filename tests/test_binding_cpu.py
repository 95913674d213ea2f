"""The Python binding's buffer checks (CPU only; no GPU and no device call).

The binding hands the library raw addresses; before it does, every torch
tensor or numpy array is checked for its device, dtype, contiguity and
element count, so that a wrong buffer raises on the host instead of being
read or written past its end on the device.  A stub stands in for the
library, so the tests also see what the binding passes on."""
import numpy as np
import pytest
import torch

import transformer_lm_step_gpt_b300 as tl
from transformer_lm_step_gpt_b300 import _buf


class StubLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def f(*args):
            self.calls.append((name, args))
            return 0
        return f


def stub_model(B=2, T=8):
    m = tl.Model.__new__(tl.Model)   # no gpt2_build: nothing touches a device
    m._lib, m._h, m.B, m.T = StubLib(), 1234, B, T
    return m


def test_buf_accepts_a_matching_host_buffer_and_passes_raw_addresses():
    a = np.zeros(16, np.int32)
    assert _buf(a, 16, "int32", "host", "a") == a.ctypes.data
    t = torch.zeros(16, dtype=torch.int32)
    assert _buf(t, 12, "int32", "host", "t") == t.data_ptr()     # more elements than needed is fine
    assert _buf(None, 16, "int32", "host", "x") is None
    assert _buf(0x1000, 16, "int32", "cuda", "x") == 0x1000       # a raw address is not checked


@pytest.mark.parametrize("x,where,err,msg", [
    (np.zeros(15, np.int32), "host", ValueError, "15 elements, need 16"),
    (np.zeros(16, np.int64), "host", TypeError, "dtype int64, need int32"),
    (np.zeros((4, 8), np.int32)[:, ::2], "host", ValueError, "contiguous"),
    (torch.zeros(16, dtype=torch.int32), "cuda", ValueError, "need a CUDA tensor"),
    (np.zeros(16, np.int32), "cuda", ValueError, "not a numpy array"),
    ([0] * 16, "host", TypeError, "unsupported buffer type list"),
    (torch.zeros(32, dtype=torch.int32)[::2], "host", ValueError, "contiguous"),
])
def test_buf_rejects_a_wrong_buffer(x, where, err, msg):
    with pytest.raises(err, match=msg):
        _buf(x, 16, "int32", where, "x")


def test_forward_host_checks_then_passes_the_addresses():
    m = stub_model()
    tok, tgt = np.zeros((2, 8), np.int32), np.ones((2, 8), np.int32)
    m.forward_host(tok, tgt, sync=False)
    name, args = m._lib.calls[-1]
    assert name == "gpt2_forward_host" and args[1] == tok.ctypes.data and args[2] == tgt.ctypes.data
    m.forward_host(tok, None, sync=False)
    assert m._lib.calls[-1][1][2] is None
    n = len(m._lib.calls)
    with pytest.raises(ValueError, match="15 elements, need 16"):
        m.forward_host(tok.reshape(-1)[:15], None, sync=False)
    with pytest.raises(TypeError, match="int64"):
        m.forward_host(tok, tgt.astype(np.int64), sync=False)
    assert len(m._lib.calls) == n                      # nothing reached the library


def test_forward_and_decode_step_need_device_buffers():
    m = stub_model()
    with pytest.raises(ValueError, match="CUDA"):
        m.forward(torch.zeros((2, 8), dtype=torch.int32), None, sync=False)
    with pytest.raises(ValueError, match="CUDA"):
        m.forward(np.zeros((2, 8), np.int32), None, sync=False)
    with pytest.raises(ValueError, match="CUDA"):
        m.decode_step(torch.zeros(2, dtype=torch.int32), 0, 1.0, torch.zeros(2), out=torch.zeros(2, dtype=torch.int32))
    assert m._lib.calls == []
    m.forward(0x10000, None, sync=False)               # raw device addresses pass through
    assert m._lib.calls[-1][0] == "gpt2_forward"


def test_layernorm_noalloc_checks_every_buffer():
    saved, tl._lib = tl._lib, StubLib()                # the module-level library, stubbed
    try:
        N, C = 4, 8
        bufs = dict(dinp=N * C, dweight=C, dbias=C, dinp_colsum=C, dout=N * C, inp=N * C, weight=C, mean=N, rstd=N)
        good = {k: torch.zeros(n) for k, n in bufs.items()}
        with pytest.raises(ValueError, match="dinp: need a CUDA tensor"):
            tl.layernorm_backward_noalloc(**good, N=N, C=C)
        raw = {k: 0x1000 * (i + 1) for i, k in enumerate(bufs)}
        tl.layernorm_backward_noalloc(**raw, N=N, C=C)
        name, args = tl._lib.calls[-1]
        assert name == "gpt2_layernorm_backward_noalloc" and args[:9] == tuple(raw.values())
    finally:
        tl._lib = saved


def test_fp8_entry_points_check_their_operands():
    with pytest.raises(ValueError, match="x: need a CUDA tensor"):
        tl.fp8_quantize(torch.zeros(16))
    q = torch.zeros((16, 32), dtype=torch.uint8)
    s = torch.ones(2)
    with pytest.raises(ValueError, match="qa: need a CUDA tensor"):
        tl.fp8_matmul(q, s, q, s)
    with pytest.raises(TypeError, match="out_dtype"):
        tl.fp8_matmul(q, s, q, s, out_dtype=torch.float16)


def test_copy_in_checks_the_length():
    m = stub_model()                                   # the stub reports an arena of 0 values
    with pytest.raises(ValueError, match="5 values, the arena holds 0"):
        m.copy_in(np.zeros(5, np.float32))
    assert not any(c[0] == "gpt2_copy_in" for c in m._lib.calls)
