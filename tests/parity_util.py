"""Shared helpers of the GPU parity tests: run the library and the CPU oracle
on the same seeded inputs and compare per tensor.

Tolerances (the method's statement of parity):
  fp32 mode  loss |delta| <= 1e-4, per-tensor relative L2 <= 1e-3
  bf16 mode  loss |delta| <= 2e-2, per-tensor relative L2 <= 2e-2
relative L2 = ||gpu - ref||_2 / max(||ref||_2, 1e-12).
"""
import numpy as np
import torch

import oracle
from transformer_lm_step_gpt_b300 import GRADS, ADAM_M, ADAM_V, PARAMS, Model, synthetic

TOL = {"fp32": dict(loss=1e-4, rel=1e-3), "bf16": dict(loss=2e-2, rel=2e-2)}


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-12))


def cuda_ids(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.int32)).cuda()


def per_tensor_errors(tab, gpu, ref, V=None, C=None):
    """{name: rel L2}; wte is compared on its V real rows only."""
    out = {}
    for name, off, n in tab:
        a, b = gpu[off:off + n], ref[off:off + n]
        if name == "wte" and V is not None:
            a, b = a[:V * C], b[:V * C]
        out[name] = rel_l2(a, b)
    return out


def run_steps(shape, precision, steps, lr, b1, b2, eps, wd, dist="uniform", seed=1234,
              kind="perturbed", check_grads_every_step=False):
    """Run `steps` training steps on the GPU and in the fp32 oracle from the
    same parameters and batches; return a dict of per-step comparisons."""
    L, C, NH, V, Vp, maxT, B, T = shape
    cfg = oracle.cfg8(*shape)
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision=precision, seed=seed)
    tab = m.tensor_table()
    assert tab == oracle.param_table(cfg)
    p0 = synthetic.params(tab, L, C, V, seed, kind=kind)
    m.copy_in(p0, PARAMS)
    po = p0.copy()
    mo = np.zeros_like(po)
    vo = np.zeros_like(po)
    res = dict(loss_gpu=[], loss_ref=[], grad_err=[], m=m, tab=tab)
    for s in range(1, steps + 1):
        tok, tgt = synthetic.batch(seed + s, B, T, V, dist)
        lg = m.forward(cuda_ids(tok), cuda_ids(tgt))
        m.zero_grad()
        m.backward()
        if s == 1 or check_grads_every_step:
            g = m.copy_out(GRADS)
        m.adamw_step(lr, b1, b2, eps, wd, s)
        lr_, g_ref, _ = oracle.step(cfg, po, mo, vo, tok, tgt, lr, b1, b2, eps, wd, s)
        res["loss_gpu"].append(lg)
        res["loss_ref"].append(lr_)
        if s == 1 or check_grads_every_step:
            res["grad_err"].append(per_tensor_errors(tab, g, g_ref, V, C))
            if s == 1:
                res["grads_gpu"], res["grads_ref"] = g, g_ref
    res["params_gpu"] = m.copy_out(PARAMS)
    res["params_ref"] = po
    res["m_gpu"], res["m_ref"] = m.copy_out(ADAM_M), mo
    res["v_gpu"], res["v_ref"] = m.copy_out(ADAM_V), vo
    return res


def assert_parity(res, shape, precision):
    L, C, NH, V, Vp, maxT, B, T = shape
    tol = TOL[precision]
    tab = res["tab"]
    for s, (a, b) in enumerate(zip(res["loss_gpu"], res["loss_ref"])):
        assert abs(a - b) <= tol["loss"], ("loss", s + 1, a, b)
    for s, errs in enumerate(res["grad_err"]):
        bad = {k: v for k, v in errs.items() if not v <= tol["rel"]}
        assert not bad, ("grad rel L2", s + 1, bad)
    # The key bias (qkvb[l, C:2C]) has an exactly zero gradient: adding a
    # constant to every key shifts all scores of a query row equally and the
    # softmax cancels it.  Its computed gradient is rounding noise, which the
    # t=1 Adam step g/(|g|+eps) turns into +-lr, so its updated value is not
    # determined by the method: it is checked separately (zero gradient,
    # |update| <= lr) and left out of the updated-parameter L2.
    qoff = dict((n, o) for n, o, _ in tab)["qkvb"]
    kb = np.concatenate([np.arange(qoff + l * 3 * C + C, qoff + l * 3 * C + 2 * C) for l in range(L)])
    qb = kb - C
    g = res["grads_gpu"]
    assert np.linalg.norm(g[kb]) <= 1e-2 * max(np.linalg.norm(g[qb]), 1e-12)
    for key in ("params", "m", "v"):
        gpu, ref = res[key + "_gpu"].copy(), res[key + "_ref"].copy()
        if key == "params":
            gpu[kb] = 0.0
            ref[kb] = 0.0
        errs = per_tensor_errors(tab, gpu, ref, V, C)
        bad = {k: v for k, v in errs.items() if not v <= tol["rel"]}
        assert not bad, (key, bad)
    # pad rows of wte: zero gradient, and they stay exactly zero
    off = tab[0][1]
    assert np.all(res["grads_gpu"][off + V * C: off + Vp * C] == 0)
    assert np.all(res["params_gpu"][off + V * C: off + Vp * C] == 0)
