"""GPU parity of generation with the key/value cache (gpt2_decode_step)
against the oracle's incremental forward and sampling rule, through the C ABI.

The library's next tokens are compared with the oracle's where the draw is
unique (the uniform is not within the tolerance of a CDF boundary) and
checked for validity against the oracle's CDF everywhere.  Teacher forcing
(the oracle's tokens fed to both sides) keeps the two sequences aligned, so
every step's scores can be compared element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from transformer_lm_step_gpt_b300 import GPT2Error, Model, synthetic
from parity_util import TOL, cuda_ids, rel_l2

pytestmark = pytest.mark.gpu

#        L  C   NH  V    Vp   maxT B  T
HS64 = (2, 128, 2, 97, 104, 64, 3, 40)      # head size 64: tensor-core prefill in bf16
HS16 = (2, 64, 4, 250, 256, 48, 2, 33)      # head size 16, ragged T
HS64_B1 = (2, 128, 2, 97, 104, 64, 1, 40)   # one sequence
GPT2_124M = (12, 768, 12, 50257, 50304, 1024)
# CDF tolerance of the validity check: the scores' error through softmax
CDF_TOL = {"fp32": 1e-4, "bf16": 5e-2}


def softmax_cdf(l, temperature):
    l = np.asarray(l, np.float64)
    if temperature <= 0:
        return None
    p = np.exp((l - l.max()) / temperature)
    return np.cumsum(p) / p.sum()


def check_draw(g, lref, temperature, u, tol, exact_when_clear=True):
    """g: the library's token; lref: the oracle's scores [V]."""
    V = lref.size
    assert 0 <= g < V
    if temperature <= 0:
        assert lref[g] >= lref.max() - tol * max(1.0, abs(lref.max()))
        if exact_when_clear:
            top2 = np.sort(lref)[-2:]
            if top2[1] - top2[0] > tol * max(1.0, abs(top2[1])):
                assert g == int(np.argmax(lref))
        return
    cdf = softmax_cdf(lref, temperature)
    lo = cdf[g - 1] if g > 0 else 0.0
    assert lo - tol <= u <= cdf[g] + tol, (g, lo, cdf[g], u)
    want = int(np.searchsorted(cdf, u, side="right"))
    if exact_when_clear and np.abs(cdf - u).min() > tol:
        assert g == want


def setup(shape, prec, seed=5):
    L, C, NH, V, Vp, maxT, B, T = shape
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision=prec, seed=seed)
    p = synthetic.params(m.tensor_table(), L, C, V, seed, kind="perturbed")
    m.copy_in(p)
    return m, p


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
@pytest.mark.parametrize("shape", [HS64, HS16])
def test_teacher_forced_decode_matches_oracle(shape, prec):
    L, C, NH, V, Vp, maxT, B, T = shape
    m, p = setup(shape, prec)
    cfg = oracle.cfg8(*shape)
    rng = np.random.default_rng(11)
    T0, n_new, temp = 9, T - 9 + 1, 0.9   # runs up to the last cache row T - 1
    prompt = rng.integers(0, V, (B, T0)).astype(np.int32)
    u = rng.random((n_new, B))
    toks_ref, lg_ref = oracle.generate(cfg, p.astype(np.float64), prompt, n_new, temp, u)
    padded = np.zeros((B, T), np.int32)
    padded[:, :T0] = prompt
    m.forward(cuda_ids(padded), None)
    u_d = torch.from_numpy(u.astype(np.float32)).cuda()
    tol = TOL[prec]["rel"]
    for i in range(n_new):
        pos = T0 - 1 + i
        tok_d = cuda_ids(toks_ref[:, pos])   # the oracle's token at this position
        nxt = m.decode_step(tok_d, pos, temp, u_d[i])
        lg = m.decode_logits()
        assert np.all(lg[:, V:] == 0)
        assert rel_l2(lg[:, :V], lg_ref[i]) <= tol, (i, rel_l2(lg[:, :V], lg_ref[i]))
        g = nxt.cpu().numpy()
        for b in range(B):
            check_draw(int(g[b]), lg_ref[i, b], temp, float(np.float32(u[i, b])), CDF_TOL[prec])


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
@pytest.mark.parametrize("shape", [HS64, HS64_B1])
def test_generate_matches_oracle(prec, shape):
    L, C, NH, V, Vp, maxT, B, T = shape
    m, p = setup(shape, prec, seed=8)
    cfg = oracle.cfg8(*shape)
    rng = np.random.default_rng(2)
    prompt = rng.integers(0, V, (B, 5)).astype(np.int32)
    n_new = 12
    u = rng.random((n_new, B)).astype(np.float32)
    got = m.generate(prompt, n_new, temperature=1.0, uniforms=u)
    want, lg_ref = oracle.generate(cfg, p.astype(np.float64), prompt, n_new, 1.0, u.astype(np.float64))
    assert got.shape == want.shape
    assert np.array_equal(got[:, :5], prompt)
    # free running: sequences agree up to the first draw that is not unique
    for b in range(B):
        for i in range(n_new):
            if got[b, 5 + i] != want[b, 5 + i]:
                cdf = softmax_cdf(lg_ref[i, b], 1.0)
                assert np.abs(cdf - u[i, b]).min() <= CDF_TOL[prec], (b, i)
                break


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_greedy_decode(prec):
    shape = HS16
    L, C, NH, V, Vp, maxT, B, T = shape
    m, p = setup(shape, prec, seed=9)
    cfg = oracle.cfg8(*shape)
    prompt = np.array([[3], [7]], np.int32)    # one-token prompts: decoding starts at position 0
    n_new = 6
    u = np.zeros((n_new, B))
    want, lg_ref = oracle.generate(cfg, p.astype(np.float64), prompt, n_new, 0.0, u)
    padded = np.zeros((B, T), np.int32)
    padded[:, :1] = prompt
    m.forward(cuda_ids(padded), None)
    u_d = torch.zeros(B, dtype=torch.float32, device="cuda")
    for i in range(n_new):
        nxt = m.decode_step(cuda_ids(want[:, i]), i, 0.0, u_d)
        g = nxt.cpu().numpy()
        for b in range(B):
            check_draw(int(g[b]), lg_ref[i, b], 0.0, 0.0, 1e-4 if prec == "fp32" else 2e-2)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_decode_row_equals_forward_row(prec):
    # the incremental row pos equals row pos of the full forward (same tokens)
    shape = HS64
    L, C, NH, V, Vp, maxT, B, T = shape
    m, _ = setup(shape, prec, seed=12)
    tok, _ = synthetic.batch(3, B, T, V)
    m.forward(cuda_ids(tok), None)
    full = m.logits().reshape(B, T, Vp)
    u_d = torch.zeros(B, dtype=torch.float32, device="cuda")
    for pos in (T - 1, 17, 0):
        m.forward(cuda_ids(tok), None)        # restore the cache rows
        m.decode_step(cuda_ids(tok[:, pos]), pos, 1.0, u_d)
        got = m.decode_logits()
        assert rel_l2(got, full[:, pos]) <= TOL[prec]["rel"], pos


def test_decode_state_and_argument_errors():
    shape = HS16
    L, C, NH, V, Vp, maxT, B, T = shape
    m, _ = setup(shape, "fp32")
    t = torch.zeros(B, dtype=torch.int32, device="cuda")
    u = torch.zeros(B, dtype=torch.float32, device="cuda")
    with pytest.raises(GPT2Error) as e:
        m.decode_step(t, 0, 1.0, u)            # no cache yet
    assert e.value.code == -4
    with pytest.raises(GPT2Error) as e:
        m.decode_logits()
    assert e.value.code == -4
    tok, tgt = synthetic.batch(1, B, T, V)
    m.forward(cuda_ids(tok), None)
    for pos in (-1, T):
        with pytest.raises(GPT2Error) as e:
            m.decode_step(t, pos, 1.0, u)
        assert e.value.code == -1
    with pytest.raises(GPT2Error) as e:
        m.decode_step(t, 0, float("nan"), u)
    assert e.value.code == -1
    m.decode_step(t, 3, 1.0, u)
    with pytest.raises(GPT2Error) as e:        # the training activations are gone
        m.backward()
    assert e.value.code == -4
    m.forward(cuda_ids(tok), cuda_ids(tgt))
    m.zero_grad()
    m.backward()
    m.adamw_step(1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    with pytest.raises(GPT2Error) as e:        # the cache holds the old weights
        m.decode_step(t, 0, 1.0, u)
    assert e.value.code == -4
    bad = torch.full((B,), V, dtype=torch.int32, device="cuda")
    m.forward(cuda_ids(tok), None)
    m.decode_step(bad, 0, 1.0, u)
    with pytest.raises(GPT2Error) as e:        # an id outside [0, V) surfaces at the next sync
        m.synchronize()
    assert e.value.code == -5


def test_gpt2_124m_decode_at_the_last_position():
    # full model shape, decode row 1023 against the forward's row 1023
    L, C, NH, V, Vp, maxT = GPT2_124M
    B, T = 2, 1024
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=21)
    tok, _ = synthetic.batch(5, B, T, V, "zipf")
    m.forward(cuda_ids(tok), None)
    full = m.logits().reshape(B, T, Vp)
    u_d = torch.full((B,), 0.5, dtype=torch.float32, device="cuda")
    for pos in (T - 1, 600):
        m.forward(cuda_ids(tok), None)
        nxt = m.decode_step(cuda_ids(tok[:, pos]), pos, 1.0, u_d).cpu().numpy()
        got = m.decode_logits()
        assert rel_l2(got[:, :V], full[:, pos, :V]) <= TOL["bf16"]["rel"], pos
        for b in range(B):
            check_draw(int(nxt[b]), full[b, pos, :V].astype(np.float64), 1.0, 0.5, CDF_TOL["bf16"],
                       exact_when_clear=False)
