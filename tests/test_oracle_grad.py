"""Whole-model pins of the oracle (CPU only).

- Central finite differences in double on tiny models, every parameter
  tensor: the gradient-checking method femtoGPT's write-up describes
  ("femtoGPT: a minimal generative pretrained Transformer in pure Rust",
  section "Gradient checking").
- The same model assembled from torch float64 library ops (embedding,
  layer_norm, linear, scaled_dot_product_attention, tanh-GELU,
  cross_entropy) with autograd: loss and every gradient.
- The fp32 oracle against the fp64 oracle.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from transformer_lm_step_gpt_b300 import synthetic

TINY = [  # (L, C, NH, V, Vp, maxT, B, T)
    (1, 8, 2, 11, 16, 8, 2, 5),
    (2, 16, 2, 32, 32, 8, 2, 8),
]


def _setup(shape, seed=0):
    L, C, NH, V, Vp, maxT, B, T = shape
    cfg = oracle.cfg8(*shape)
    tab = oracle.param_table(cfg)
    # perturbed: non-trivial biases and LayerNorm gamma/beta exercise every term
    p = synthetic.params(tab, L, C, V, seed, kind="perturbed", dtype=np.float64)
    # larger weights than the GPT-2 init make every path matter numerically
    p *= 5.0
    for name, off, n in tab:
        if name in ("ln1w", "ln2w", "lnfw"):
            p[off:off + n] = 1.0 + (p[off:off + n] / 5.0 - 1.0)
    tok, tgt = synthetic.batch(seed + 1, B, T, V)
    return cfg, tab, p, tok, tgt


@pytest.mark.parametrize("shape", TINY)
def test_finite_difference_every_tensor(shape):
    cfg, tab, p, tok, tgt = _setup(shape)
    L, C, NH, V, Vp, maxT, B, T = shape
    r = oracle.fwdbwd(cfg, p, tok, tgt)
    g = r["grads"]
    rng = np.random.default_rng(1)
    h = 1e-5
    for name, off, n in tab:
        idx = rng.choice(n, size=min(n, 12), replace=False) + off
        if name == "wte":  # make sure token rows (not only pad rows) are sampled
            rows = np.unique(tok)[:3]
            idx = np.concatenate([idx, rows * C + off, rows * C + off + C - 1])
        for e in idx:
            pp = p.copy(); pp[e] += h
            pm = p.copy(); pm[e] -= h
            lp = oracle.fwdbwd(cfg, pp, tok, tgt, want_grads=False)["loss"]
            lm = oracle.fwdbwd(cfg, pm, tok, tgt, want_grads=False)["loss"]
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[e]) <= 1e-6 * max(abs(fd), 1e-3), (name, e - off, fd, g[e])
    # pad rows of wte and unused positions of wpe get exactly zero gradient
    wte_off = tab[0][1]
    assert np.all(g[wte_off + V * C: wte_off + Vp * C] == 0)
    wpe_off = tab[1][1]
    assert np.all(g[wpe_off + T * C: wpe_off + maxT * C] == 0)


def torch_reference_loss(shape, tab, p, tok, tgt):
    L, C, NH, V, Vp, maxT, B, T = shape
    hs = C // NH
    P = {name: torch.tensor(p[off:off + n], dtype=torch.float64, requires_grad=True)
         for name, off, n in tab}
    wte = P["wte"].view(Vp, C)
    wpe = P["wpe"].view(maxT, C)
    tk = torch.tensor(tok, dtype=torch.long)
    x = F.embedding(tk, wte) + wpe[:T]
    for l in range(L):
        h = F.layer_norm(x, (C,), P["ln1w"].view(L, C)[l], P["ln1b"].view(L, C)[l], eps=1e-5)
        qkv = F.linear(h, P["qkvw"].view(L, 3 * C, C)[l], P["qkvb"].view(L, 3 * C)[l])
        q, k, v = qkv.split(C, dim=-1)
        sh = lambda z: z.view(B, T, NH, hs).transpose(1, 2)
        y = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
        y = y.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, P["attprojw"].view(L, C, C)[l], P["attprojb"].view(L, C)[l])
        h2 = F.layer_norm(x, (C,), P["ln2w"].view(L, C)[l], P["ln2b"].view(L, C)[l], eps=1e-5)
        f = F.gelu(F.linear(h2, P["fcw"].view(L, 4 * C, C)[l], P["fcb"].view(L, 4 * C)[l]),
                   approximate="tanh")
        x = x + F.linear(f, P["fcprojw"].view(L, C, 4 * C)[l], P["fcprojb"].view(L, C)[l])
    xf = F.layer_norm(x, (C,), P["lnfw"], P["lnfb"], eps=1e-5)
    logits = F.linear(xf, wte[:V])
    loss = F.cross_entropy(logits.reshape(-1, V), torch.tensor(tgt, dtype=torch.long).reshape(-1))
    return loss, P


@pytest.mark.parametrize("shape", TINY + [(3, 24, 4, 50, 64, 16, 3, 16), (0, 8, 2, 13, 16, 6, 2, 6)])
def test_whole_model_vs_torch_autograd(shape):
    cfg, tab, p, tok, tgt = _setup(shape, seed=3)
    r = oracle.fwdbwd(cfg, p, tok, tgt)
    loss, P = torch_reference_loss(shape, tab, p, tok, tgt)
    loss.backward()
    assert abs(r["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
    for name, off, n in tab:
        ref = P[name].grad.numpy() if P[name].grad is not None else np.zeros(n)
        ours = r["grads"][off:off + n]
        err = np.linalg.norm(ours - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err < 1e-10, (name, err)


def test_f32_oracle_close_to_f64():
    shape = (2, 64, 4, 256, 256, 32, 4, 32)
    L, C, NH, V, Vp, maxT, B, T = shape
    cfg = oracle.cfg8(*shape)
    tab = oracle.param_table(cfg)
    p = synthetic.params(tab, L, C, V, 5, kind="perturbed", dtype=np.float64)
    tok, tgt = synthetic.batch(6, B, T, V)
    r64 = oracle.fwdbwd(cfg, p, tok, tgt)
    r32 = oracle.fwdbwd(cfg, p.astype(np.float32), tok, tgt)
    assert abs(r32["loss"] - r64["loss"]) < 1e-5
    for name, off, n in tab:
        a, b = r32["grads"][off:off + n], r64["grads"][off:off + n]
        err = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
        assert err < 1e-5, (name, err)


def test_step_matches_torch_adamw():
    shape = TINY[1]
    cfg, tab, p, tok, tgt = _setup(shape, seed=9)
    loss, P = torch_reference_loss(shape, tab, p, tok, tgt)
    loss.backward()
    opt = torch.optim.AdamW(list(P.values()), lr=1e-2, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.1)
    opt.step()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    pp = p.copy()
    oracle.step(cfg, pp, m, v, tok, tgt, 1e-2, 0.9, 0.999, 1e-8, 0.1, 1)
    for name, off, n in tab:
        np.testing.assert_allclose(pp[off:off + n], P[name].detach().numpy(), rtol=1e-9, atol=1e-12)
