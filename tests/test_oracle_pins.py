"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test checks the oracle against a number the pages print, a closed form,
an invariant, a special case that reduces to a library routine (torch float64
CPU ops, numpy), or a published known-answer vector.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                out[k] = v
    return out


# ---- printed counters of the run log ---------------------------------------

def test_num_parameters_matches_run_log():
    g = _golden("run_log_124M.txt")
    L, C, NH = int(g["num_layers"][0]), int(g["channels"][0]), int(g["num_heads"][0])
    V, maxT = int(g["vocab_size"][0]), int(g["max_seq_len"][0])
    cfg = oracle.cfg8(L, C, NH, V, V, maxT, 4, 64)
    assert oracle.num_params(cfg) == int(g["num_parameters"][0])
    # the parameter array is one contiguous 1-D block: tensors tile it exactly
    tab = oracle.param_table(cfg)
    off = 0
    for _, o, n in tab:
        assert o == off
        off += n
    assert off == oracle.num_params(cfg)


def test_num_activations_matches_run_log_shape():
    g = _golden("run_log_124M.txt")
    L, C, NH = int(g["num_layers"][0]), int(g["channels"][0]), int(g["num_heads"][0])
    V, maxT = int(g["vocab_size"][0]), int(g["max_seq_len"][0])
    bt = int(g["train_tokens"][0]) // int(g["train_num_batches"][0])
    assert bt == 256 and int(g["val_tokens"][0]) // int(g["val_num_batches"][0]) == 256
    want = int(g["num_activations"][0])
    hits = []
    for B in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        T = bt // B
        if oracle.num_activations(oracle.cfg8(L, C, NH, V, V, maxT, B, T)) == want:
            hits.append((B, T))
    # exactly one split of B*T = 256 reproduces the printed count
    assert hits == [(4, 64)]


def test_padded_vocab_param_count():
    # Vp = 50304 pads 47 rows of wte: 47 * 768 more parameters
    base = oracle.num_params(oracle.cfg8(12, 768, 12, 50257, 50257, 1024, 4, 64))
    pad = oracle.num_params(oracle.cfg8(12, 768, 12, 50257, 50304, 1024, 4, 64))
    assert pad - base == 47 * 768 == 124475904 - 124439808


# ---- GELU -------------------------------------------------------------------

def test_gelu_constants_and_definition():
    g = _golden("gelu_constants.txt")
    s, a = float(g["tanh_scale"][0]), float(g["cubic_coeff"][0])
    assert abs(s - math.sqrt(2 / math.pi)) < 1e-7
    x = np.linspace(-6, 6, 2001)
    y = oracle.gelu_forward(x)
    exact = x * 0.5 * (1 + np.array([math.erf(v / math.sqrt(2)) for v in x]))
    assert np.max(np.abs(y - exact)) < 1e-3          # tanh form ~ x * Phi(x)
    # the printed (truncated) macro agrees with the full-precision constant
    printed = x / 2 * (1 + np.tanh(s * (x + a * x ** 3)))
    assert np.max(np.abs(y - printed)) < 1e-7
    assert oracle.gelu_forward(np.array([0.0]))[0] == 0.0
    big = oracle.gelu_forward(np.array([20.0, -20.0]))
    assert abs(big[0] - 20.0) < 1e-12 and abs(big[1]) < 1e-12


def test_gelu_vs_torch_tanh_gelu():
    x = torch.linspace(-8, 8, 4097, dtype=torch.float64, requires_grad=True)
    y = F.gelu(x, approximate="tanh")
    ours = oracle.gelu_forward(x.detach().numpy())
    np.testing.assert_allclose(ours, y.detach().numpy(), rtol=1e-13, atol=1e-15)
    dout = torch.randn(4097, dtype=torch.float64, generator=torch.Generator().manual_seed(0))
    y.backward(dout)
    d = oracle.gelu_backward(x.detach().numpy(), dout.numpy())
    np.testing.assert_allclose(d, x.grad.numpy(), rtol=1e-12, atol=1e-13)


# ---- LayerNorm ---------------------------------------------------------------

def test_layernorm_vs_torch_and_special_cases():
    rng = np.random.default_rng(1)
    N, C = 7, 24
    x = rng.normal(size=(N, C)) * 3 + 1
    w = rng.normal(size=C)
    b = rng.normal(size=C)
    y, mean, rstd = oracle.layernorm_forward(x, w, b)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    yt = F.layer_norm(xt, (C,), wt, bt, eps=1e-5)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mean, x.mean(1), rtol=1e-13)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(x.var(1) + 1e-5), rtol=1e-12)
    dy = rng.normal(size=(N, C))
    yt.backward(torch.tensor(dy))
    dx, dw, db = oracle.layernorm_backward(dy, x, w, mean, rstd)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-10, atol=1e-12)
    # constant rows: output is beta; with xhat = 0 the input gradient reduces
    # to the closed form (g - mean(g)) / sqrt(eps), g = dy * gamma
    xc = np.full((3, C), 2.5)
    yc, _, rc = oracle.layernorm_forward(xc, w, b)
    np.testing.assert_allclose(yc, np.broadcast_to(b, (3, C)), atol=1e-12)
    np.testing.assert_allclose(rc, 1 / math.sqrt(1e-5), rtol=1e-14)
    dyc = rng.normal(size=(3, C))
    dxc, _, dbc = oracle.layernorm_backward(dyc, xc, w, np.full(3, 2.5), rc)
    gc = dyc * w
    np.testing.assert_allclose(dxc, (gc - gc.mean(1, keepdims=True)) / math.sqrt(1e-5), rtol=1e-11)
    np.testing.assert_allclose(dbc, dyc.sum(0), rtol=1e-13)
    # gamma = 1, beta = 0: zero mean, unit (biased) variance up to eps
    y1, _, _ = oracle.layernorm_forward(x, np.ones(C), np.zeros(C))
    np.testing.assert_allclose(y1.mean(1), 0, atol=1e-12)
    np.testing.assert_allclose(y1.var(1), x.var(1) / (x.var(1) + 1e-5), rtol=1e-12)


# ---- Linear ------------------------------------------------------------------

def test_matmul_identity_and_numpy():
    rng = np.random.default_rng(2)
    N, IC, OC = 5, 9, 9
    x = rng.normal(size=(N, IC))
    bias = rng.normal(size=OC)
    np.testing.assert_allclose(oracle.matmul_forward(x, np.eye(IC), bias), x + bias, rtol=1e-15)
    OC = 13
    W = rng.normal(size=(OC, IC))
    bias = rng.normal(size=OC)
    np.testing.assert_allclose(oracle.matmul_forward(x, W, bias), x @ W.T + bias, rtol=1e-12)
    np.testing.assert_allclose(oracle.matmul_forward(x, W), x @ W.T, rtol=1e-12)
    dout = rng.normal(size=(N, OC))
    dx, dW, db = oracle.matmul_backward(dout, x, W)
    np.testing.assert_allclose(dx, dout @ W, rtol=1e-12)
    np.testing.assert_allclose(dW, dout.T @ x, rtol=1e-12)
    np.testing.assert_allclose(db, dout.sum(0), rtol=1e-12)


# ---- attention ----------------------------------------------------------------

def _sdpa(qkv, B, T, C, NH):
    hs = C // NH
    q, k, v = qkv.split(C, dim=-1)
    sh = lambda z: z.view(B, T, NH, hs).transpose(1, 2)
    y = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
    return y.transpose(1, 2).reshape(B, T, C)


@pytest.mark.parametrize("B,T,C,NH", [(2, 8, 16, 2), (1, 5, 12, 3), (3, 1, 8, 2),
                                      # every head size the library accepts: 16, 32, 64, 128
                                      (1, 7, 64, 4), (2, 6, 64, 2), (1, 9, 128, 2), (1, 5, 128, 1)])
def test_attention_vs_torch_sdpa(B, T, C, NH):
    rng = np.random.default_rng(3)
    qkv = rng.normal(size=(B, T, 3 * C))
    y, pre, att = oracle.attention_forward(qkv, B, T, C, NH)
    qt = torch.tensor(qkv, requires_grad=True)
    yt = _sdpa(qt, B, T, C, NH)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-13)
    # rows of P sum to one and vanish above the diagonal
    np.testing.assert_allclose(att.sum(-1), 1.0, rtol=1e-14)
    assert np.all(np.triu(att, 1) == 0)
    dy = rng.normal(size=(B, T, C))
    yt.backward(torch.tensor(dy))
    dqkv = oracle.attention_backward(dy, qkv, att, B, T, C, NH)
    np.testing.assert_allclose(dqkv, qt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    B, T, C, NH = 1, 6, 8, 2
    qkv = rng.normal(size=(B, T, 3 * C))
    y, _, att = oracle.attention_forward(qkv, B, T, C, NH)
    # row 0 attends only to itself: y_0 = v_0
    np.testing.assert_allclose(y[0, 0], qkv[0, 0, 2 * C:], rtol=1e-14)
    # equal keys: uniform weights 1/(i+1), y_i = mean of v_0..v_i
    qkv2 = qkv.copy()
    qkv2[0, :, C:2 * C] = qkv2[0, 0, C:2 * C]
    y2, _, att2 = oracle.attention_forward(qkv2, B, T, C, NH)
    for i in range(T):
        np.testing.assert_allclose(att2[0, :, i, :i + 1], 1.0 / (i + 1), rtol=1e-14)
        np.testing.assert_allclose(y2[0, i], qkv2[0, :i + 1, 2 * C:].mean(0), rtol=1e-12)
    # T = 1: output equals v
    y1, _, _ = oracle.attention_forward(qkv[:, :1], B, 1, C, NH)
    np.testing.assert_allclose(y1[0, 0], qkv[0, 0, 2 * C:], rtol=1e-14)


# ---- softmax / cross-entropy ---------------------------------------------------

def test_crossentropy_vs_torch_and_closed_forms():
    rng = np.random.default_rng(5)
    N, V = 9, 37
    logits = rng.normal(size=(N, V)) * 4
    tg = rng.integers(0, V, N).astype(np.int32)
    losses, probs = oracle.crossentropy_forward(logits, tg)
    np.testing.assert_allclose(probs.sum(1), 1.0, rtol=1e-14)
    lt = torch.tensor(logits, requires_grad=True)
    ref = F.cross_entropy(lt, torch.tensor(tg, dtype=torch.long), reduction="none")
    np.testing.assert_allclose(losses, ref.detach().numpy(), rtol=1e-13)
    ref.mean().backward()
    d = oracle.crossentropy_backward(probs, tg, 1.0 / N)
    np.testing.assert_allclose(d, lt.grad.numpy(), rtol=1e-12, atol=1e-15)
    # all-zero logits: loss is exactly ln V and dlogits = (1/V - onehot) / N
    z_losses, z_probs = oracle.crossentropy_forward(np.zeros((N, V)), tg)
    np.testing.assert_allclose(z_losses, math.log(V), rtol=1e-15)
    dz = oracle.crossentropy_backward(z_probs, tg, 1.0 / N)
    want = np.full((N, V), 1.0 / V)
    want[np.arange(N), tg] -= 1.0
    np.testing.assert_allclose(dz, want / N, rtol=1e-14, atol=1e-18)


# ---- AdamW -----------------------------------------------------------------------

def test_adamw_closed_forms():
    rng = np.random.default_rng(6)
    n = 1000
    p0 = rng.normal(size=n)
    g = rng.normal(size=n)
    lr, eps = 1e-3, 1e-8
    # t = 1, wd = 0: mhat = g, vhat = g^2 -> p1 = p0 - lr * g / (|g| + eps)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    oracle.adamw(p, g, m, v, lr, 0.9, 0.999, eps, 0.0, 1)
    np.testing.assert_allclose(p, p0 - lr * g / (np.abs(g) + eps), rtol=1e-12)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-14)
    np.testing.assert_allclose(v, 0.001 * g * g, rtol=1e-12)
    # g = 0: pure decoupled decay p1 = p0 (1 - lr wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    oracle.adamw(p, np.zeros(n), m, v, lr, 0.9, 0.999, eps, 0.1, 1)
    np.testing.assert_allclose(p, p0 * (1 - lr * 0.1), rtol=1e-15)


def test_adamw_vs_torch_optim():
    rng = np.random.default_rng(7)
    n = 513
    p0 = rng.normal(size=n)
    lr, b1, b2, eps, wd = 3e-3, 0.9, 0.95, 1e-8, 0.1
    pt = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.AdamW([pt], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 6):
        g = rng.normal(size=n)
        pt.grad = torch.tensor(g)
        opt.step()
        oracle.adamw(p, g, m, v, lr, b1, b2, eps, wd, t)
        np.testing.assert_allclose(p, pt.detach().numpy(), rtol=1e-12, atol=1e-15)


# ---- encoder -----------------------------------------------------------------------

def test_encoder_gather_and_counting():
    rng = np.random.default_rng(8)
    B, T, C, V, maxT = 3, 5, 4, 11, 8
    wte = rng.normal(size=V * C)
    wpe = rng.normal(size=maxT * C)
    tok = rng.integers(0, V, (B, T)).astype(np.int32)
    out = oracle.encoder_forward(tok, wte, wpe, B, T, C).reshape(B, T, C)
    np.testing.assert_array_equal(out, wte.reshape(V, C)[tok] + wpe.reshape(maxT, C)[:T])
    # all tokens equal: that row's gradient is the sum of every position's
    dout = rng.normal(size=(B, T, C))
    same = np.full((B, T), 7, np.int32)
    dwte, dwpe = oracle.encoder_backward(dout.reshape(-1), same, V, B, T, C, maxT)
    dwte = dwte.reshape(V, C)
    np.testing.assert_allclose(dwte[7], dout.reshape(-1, C).sum(0), rtol=1e-13)
    assert np.all(np.delete(dwte, 7, axis=0) == 0)
    np.testing.assert_allclose(dwpe.reshape(maxT, C)[:T], dout.sum(0), rtol=1e-13)
    assert np.all(dwpe.reshape(maxT, C)[T:] == 0)


# ---- init generator -----------------------------------------------------------------

def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        out = oracle.philox4x32_10(w[0:4], w[4:6])
        assert list(out) == w[6:10]


def test_init_params_distribution():
    L, C, NH, V, Vp, maxT = 2, 64, 4, 250, 256, 32
    cfg = oracle.cfg8(L, C, NH, V, Vp, maxT, 4, 32)
    p = oracle.init_params(cfg, 1337)
    tab = {n: (o, k) for n, o, k in oracle.param_table(cfg)}
    get = lambda n: p[tab[n][0]:tab[n][0] + tab[n][1]]
    wte = get("wte").reshape(Vp, C)
    assert np.all(wte[V:] == 0)
    big = np.concatenate([wte[:V].ravel(), get("wpe"), get("qkvw"), get("fcw")])
    assert abs(big.mean()) < 3 * 0.02 / math.sqrt(big.size)
    assert abs(big.std() / 0.02 - 1) < 0.02
    res = np.concatenate([get("attprojw"), get("fcprojw")])
    assert abs(res.std() / (0.02 / math.sqrt(2 * L)) - 1) < 0.03
    for n in ("ln1w", "ln2w", "lnfw"):
        assert np.all(get(n) == 1.0)
    for n in ("ln1b", "ln2b", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
        assert np.all(get(n) == 0.0)
    # Box-Muller pairs: element 2k and 2k+1 share a radius
    e = tab["wpe"][0]
    e -= e % 2
    r2 = oracle.normal_at(1337, e) ** 2 + oracle.normal_at(1337, e + 1) ** 2
    assert r2 > 0


def test_initial_loss_near_ln_v():
    from transformer_lm_step_gpt_b300 import synthetic
    L, C, NH, V, maxT, B, T = 2, 64, 4, 256, 32, 4, 32
    cfg = oracle.cfg8(L, C, NH, V, V, maxT, B, T)
    p = oracle.init_params(cfg, 1337)
    tok, tgt = synthetic.batch(1338, B, T, V)
    r = oracle.fwdbwd(cfg, p, tok, tgt, want_grads=False)
    assert abs(r["loss"] - math.log(V)) < 0.05


def test_oracle_results_do_not_depend_on_the_thread_count():
    # OpenMP splits only independent outputs; every sum runs in formula order
    from transformer_lm_step_gpt_b300 import synthetic
    L, C, NH, V, Vp, maxT, B, T = 2, 32, 2, 50, 56, 16, 3, 12
    cfg = oracle.cfg8(L, C, NH, V, Vp, maxT, B, T)
    p = synthetic.params(oracle.param_table(cfg), L, C, V, 3, kind="perturbed")
    tok, tgt = synthetic.batch(4, B, T, V, "zipf")
    out = []
    try:
        for n in (1, max(2, min(8, os.cpu_count() or 2))):
            oracle.set_threads(n)
            r = oracle.fwdbwd(cfg, p, tok, tgt)
            out.append((r["loss"], r["grads"].copy()))
    finally:
        oracle.set_threads(0)
    assert out[0][0] == out[1][0]
    assert np.array_equal(out[0][1], out[1][1])
