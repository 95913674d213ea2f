"""The allocation-free LayerNorm backward (gpt2_layernorm_backward_noalloc)
against the library's existing entry point.

Some callers of this library cannot call cudaMalloc (their device memory
belongs to another allocator, or a device-synchronising allocation is not
acceptable in their loop); this entry point serves them with a static
scratch array.  Its outputs are checked against gpt2_backward: in an fp32
model, the final LayerNorm's backward produces the gradients of lnfw and
lnfb and, through its residual-gradient column sums, the fcproj bias
gradient of the last block.  The LayerNorm's inputs are reconstructed from
what the existing entry points expose (the residual stream entering LN_f,
the logits, wte and lnfw).  Two calls in a row must both match: the second
one reuses the partials the first left in the static array.  The outputs are
also compared element by element with the oracle's LayerNorm backward at the
GPT-2 widths C = 768 and 1024, with output buffers that start nonzero (the
call adds into them).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import transformer_lm_step_gpt_b300 as tl
from transformer_lm_step_gpt_b300 import GRADS, PARAMS, Model, synthetic

pytestmark = pytest.mark.gpu

SHAPE = (2, 64, 4, 250, 256, 64, 3, 50)  # L C NH V Vp maxT B T  (M = 150, ragged)
REL = 1e-3  # the fp32-mode per-tensor tolerance of the parity tests


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-12))


def test_noalloc_layernorm_backward_matches_gpt2_backward():
    L, C, NH, V, Vp, maxT, B, T = SHAPE
    M = B * T
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="fp32", seed=21)
    tab = dict((n, (o, k)) for n, o, k in m.tensor_table())
    p = synthetic.params(m.tensor_table(), L, C, V, 21, kind="perturbed")
    m.copy_in(p, PARAMS)
    tok, tgt = synthetic.batch(22, B, T, V, "zipf")
    tok_d, tgt_d = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    # existing entry points: the residual stream entering LN_f, the logits
    m.forward(tok_d, None)
    x = m.residual(L).astype(np.float64)
    logits = m.logits()[:, :V].astype(np.float64)
    # and the gradients gpt2_backward produces
    m.forward(tok_d, tgt_d)
    m.zero_grad()
    m.backward()
    g = m.copy_out(GRADS)
    want_dw = g[tab["lnfw"][0]:tab["lnfw"][0] + C]
    want_db = g[tab["lnfb"][0]:tab["lnfb"][0] + C]
    want_cs = g[tab["fcprojb"][0] + (L - 1) * C:tab["fcprojb"][0] + L * C]
    # the final LayerNorm's inputs: dout = dlogits . wte, mean and rstd of x
    z = logits - logits.max(1, keepdims=True)
    prob = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    prob[np.arange(M), tgt.reshape(-1)] -= 1.0
    wte = p[tab["wte"][0]:tab["wte"][0] + V * C].reshape(V, C).astype(np.float64)
    dout = (prob / M) @ wte
    mean = x.mean(1)
    rstd = 1.0 / np.sqrt(x.var(1) + 1e-5)
    w = p[tab["lnfw"][0]:tab["lnfw"][0] + C]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    ins = [dev(dout), dev(x), dev(w), dev(mean), dev(rstd)]
    lib = tl.load_library()
    results = []
    for _ in range(2):  # two calls in a row share the static scratch
        outs = [torch.zeros(M, C, device="cuda"), torch.zeros(C, device="cuda"),
                torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda")]
        rc = lib.gpt2_layernorm_backward_noalloc(*[t.data_ptr() for t in outs], *[t.data_ptr() for t in ins],
                                                 M, C, None)
        assert rc == 0, lib.gpt2_last_error(None)
        torch.cuda.synchronize()
        dx, dw, db, cs = [t.cpu().numpy() for t in outs]
        assert rel_l2(dw, want_dw) <= REL
        assert rel_l2(db, want_db) <= REL
        assert rel_l2(cs, want_cs) <= REL
        assert rel_l2(dx.sum(0), cs) <= 1e-5
        results.append((dx, dw, db, cs))
    for a, b in zip(results[0], results[1]):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("N,C", [(1000, 768), (2000, 1024)])
def test_noalloc_layernorm_backward_matches_the_oracle(N, C):
    rng = np.random.default_rng(N + C)
    x = rng.normal(0.3, 1.7, (N, C)).astype(np.float32)
    dout = rng.normal(0, 1e-3, (N, C)).astype(np.float32)
    w = (1.0 + rng.normal(0, 0.1, C)).astype(np.float32)
    x64 = x.astype(np.float64)
    mean = x64.mean(1).astype(np.float32)
    rstd = (1.0 / np.sqrt(x64.var(1) + 1e-5)).astype(np.float32)
    # the oracle on exactly the inputs the GPU reads
    dx_ref, dw_ref, db_ref = oracle.layernorm_backward(dout.astype(np.float64), x64, w.astype(np.float64),
                                                       mean.astype(np.float64), rstd.astype(np.float64))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()  # noqa: E731
    ins = [dev(dout), dev(x), dev(w), dev(mean), dev(rstd)]
    # outputs start nonzero: the call adds into them
    init = [rng.normal(0, 1e-3, (N, C)), rng.normal(0, 1e-2, C), rng.normal(0, 1e-2, C), rng.normal(0, 1e-2, C)]
    init = [a.astype(np.float32) for a in init]
    results = []
    for _ in range(2):
        outs = [dev(a) for a in init]
        tl.layernorm_backward_noalloc(*outs, *ins, N, C)
        tl.noalloc_check()
        dx, dw, db, cs = [t.cpu().numpy().astype(np.float64) for t in outs]
        dx -= init[0]
        dw -= init[1]
        db -= init[2]
        cs -= init[3]
        assert rel_l2(dx, dx_ref) <= REL
        assert np.max(np.abs(dx - dx_ref)) <= REL * np.max(np.abs(dx_ref))
        assert rel_l2(dw, dw_ref) <= REL
        assert rel_l2(db, db_ref) <= REL
        # the column sums of the updated dinp: of the initial values plus dx
        assert rel_l2(cs, (init[0].astype(np.float64) + dx_ref).sum(0)) <= REL
        results.append((dx, dw, db, cs))
    for a, b in zip(results[0], results[1]):
        assert np.array_equal(a, b)


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    lib = tl.load_library()
    big_n, C = 1 << 20, 1024  # ceil(N/64) * 3 * C = 3 * 2^24 floats > 2^21
    rc = lib.gpt2_layernorm_backward_noalloc(*([ctypes.c_void_p(16)] * 9), big_n, C, None)
    assert rc == -1
    assert b"static scratch" in lib.gpt2_last_error(None)
