"""Checkpoint save / resume (gpt2_save_checkpoint, gpt2_load_checkpoint):
the saved state comes back bit for bit, and a resumed model takes exactly
the same next step as the one that saved it (every kernel is
deterministic).  Inputs come from an int32 token file through TokenFile."""
import numpy as np
import pytest

import transformer_lm_step_gpt_b300 as tl
from transformer_lm_step_gpt_b300 import synthetic

SHAPE = (2, 64, 4, 250, 256, 64, 3, 48)  # L C NH V Vp maxT B T


def _model(prec, seed, shape=SHAPE):
    L, C, NH, V, Vp, maxT, B, T = shape
    return tl.Model(L, C, NH, V, Vp, maxT, B, T, precision=prec, seed=seed)


def _step(m, f, t):
    import torch
    x, y = f.next_batch(m.B, m.T)
    loss = m.forward(torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda())
    m.zero_grad()
    m.backward()
    m.adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, t)
    return loss


@pytest.mark.gpu
@pytest.mark.parametrize("prec", ["bf16", "fp32"])
def test_save_load_resume_is_exact(tmp_path, prec):
    L, C, NH, V, Vp, maxT, B, T = SHAPE
    stream = synthetic.token_stream(77, 4000, V)
    toks = tmp_path / "train.bin"
    np.asarray(stream, dtype="<i4").tofile(toks)
    a = _model(prec, seed=11)
    fa = tl.TokenFile(str(toks))
    for t in (1, 2):
        _step(a, fa, t)
    ck = tmp_path / "a.ckpt"
    a.save_checkpoint(str(ck), step=2)
    b = _model(prec, seed=12)  # different init, overwritten by the load
    assert b.load_checkpoint(str(ck)) == 2
    for arena in (tl.PARAMS, tl.ADAM_M, tl.ADAM_V):
        np.testing.assert_array_equal(a.copy_out(arena), b.copy_out(arena))
    # the file: 64 header words + 3 arenas
    assert ck.stat().st_size == 4 * 64 + 3 * 4 * a.num_params
    fb = tl.TokenFile(str(toks))
    fb.next_batch(B, T)
    fb.next_batch(B, T)  # same cursor as fa
    la = _step(a, fa, 3)
    lb = _step(b, fb, 3)
    assert la == lb
    np.testing.assert_array_equal(a.copy_out(tl.PARAMS), b.copy_out(tl.PARAMS))


@pytest.mark.gpu
def test_load_checks_shape_and_length(tmp_path):
    a = _model("bf16", seed=3)
    ck = tmp_path / "a.ckpt"
    a.save_checkpoint(str(ck), step=5)
    # precision and batch shape may differ
    L, C, NH, V, Vp, maxT, B, T = SHAPE
    c = _model("fp32", seed=4, shape=(L, C, NH, V, Vp, maxT, 2, 16))
    assert c.load_checkpoint(str(ck)) == 5
    np.testing.assert_array_equal(a.copy_out(tl.PARAMS), c.copy_out(tl.PARAMS))
    # another model shape is refused
    d = _model("bf16", seed=4, shape=(L, 128, NH, V, Vp, maxT, B, T))
    with pytest.raises(tl.GPT2Error) as e:
        d.load_checkpoint(str(ck))
    assert e.value.code == -1
    # a truncated file is refused and leaves the model as it was
    before = a.copy_out(tl.PARAMS)
    short = tmp_path / "short.ckpt"
    short.write_bytes(ck.read_bytes()[: 4 * 64 + 1000])
    with pytest.raises(tl.GPT2Error) as e:
        a.load_checkpoint(str(short))
    assert e.value.code == -8
    np.testing.assert_array_equal(a.copy_out(tl.PARAMS), before)
    with pytest.raises(tl.GPT2Error) as e:
        a.load_checkpoint(str(tmp_path / "missing.ckpt"))
    assert e.value.code == -8
