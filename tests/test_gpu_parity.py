"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs, through the C ABI.  Shapes are the method's configurations (tiny,
char-level, GPT-2 124M / 350M) plus ragged ones that leave partial tiles in
every dimension.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_lm_step_gpt_b300 import GPT2Error, GRADS, PARAMS, Model, synthetic
from parity_util import TOL, assert_parity, cuda_ids, per_tensor_errors, rel_l2, run_steps

pytestmark = pytest.mark.gpu

TINY = (2, 64, 4, 256, 256, 32, 4, 32)          # L C NH V Vp maxT B T
CHAR = (8, 128, 8, 1000, 1000, 64, 32, 64)
RAGGED = (2, 64, 4, 250, 256, 64, 3, 50)        # M=150, V<Vp, T=50, hs=16
RAGGED64 = (1, 128, 2, 1000, 1000, 96, 2, 80)   # hs=64, M=160, T=80
RAGGED64_ODD = (1, 128, 2, 1000, 1000, 200, 2, 199)  # hs=64, T=199: not a multiple of 4
RAGGED32 = (1, 64, 2, 300, 304, 48, 2, 40)      # hs=32, V<Vp, T=40
RAGGED128 = (1, 128, 1, 200, 200, 48, 2, 33)    # hs=128, one head, T=33
SINGLE_TOKEN = (1, 128, 2, 100, 104, 8, 2, 1)   # T=1 (each position attends to itself), M=2
GPT2_124M = (12, 768, 12, 50257, 50304, 1024)


def test_init_matches_oracle_generator():
    L, C, NH, V, Vp, maxT, B, T = TINY
    m = Model(L, C, NH, 250, Vp, maxT, B, T, precision="fp32", seed=4242)
    got = m.copy_out(PARAMS).astype(np.float64)
    want = oracle.init_params(oracle.cfg8(L, C, NH, 250, Vp, maxT, B, T), 4242)
    np.testing.assert_allclose(got, want.astype(np.float32), rtol=1e-6, atol=1e-9)
    tab = dict((n, (o, k)) for n, o, k in m.tensor_table())
    o, k = tab["wte"]
    assert np.all(got[o + 250 * C:o + k] == 0)


def test_encoder_gather_bit_exact():
    L, C, NH, V, Vp, maxT, B, T = TINY
    for prec in ("fp32", "bf16"):
        m = Model(L, C, NH, V, Vp, maxT, B, T, precision=prec, seed=7)
        p = synthetic.params(m.tensor_table(), L, C, V, 7, kind="perturbed")
        m.copy_in(p)
        tok, _ = synthetic.batch(8, B, T, V, "zipf")
        m.forward(cuda_ids(tok), None)
        ref = oracle.residuals_f32(oracle.cfg8(*TINY), p, tok)
        assert np.array_equal(m.residual(0), ref[0])  # bit for bit
        if prec == "fp32":
            for l in range(1, L + 1):
                assert rel_l2(m.residual(l), ref[l]) < 1e-5


def test_forward_logits_fp32():
    L, C, NH, V, Vp, maxT, B, T = RAGGED
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="fp32", seed=3)
    p = synthetic.params(m.tensor_table(), L, C, V, 3, kind="perturbed")
    m.copy_in(p)
    tok, _ = synthetic.batch(4, B, T, V)
    m.forward(cuda_ids(tok), None)
    got = m.logits()
    ref = oracle.fwdbwd(oracle.cfg8(*RAGGED), p, tok, None, want_grads=False, want_logits=True)["logits"]
    assert rel_l2(got[:, :V], ref) < 1e-5
    assert np.all(got[:, V:] == 0)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_config_tiny_one_step(prec):
    res = run_steps(TINY, prec, 1, 1e-4, 0.9, 0.999, 1e-8, 0.0, "uniform", seed=11)
    assert_parity(res, TINY, prec)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_config_char_ten_steps(prec):
    res = run_steps(CHAR, prec, 10, 3e-4, 0.9, 0.999, 1e-8, 0.1, "zipf", seed=12)
    assert_parity(res, CHAR, prec)
    # the loss curve goes down on a fixed-distribution stream
    assert res["loss_gpu"][-1] < res["loss_gpu"][0]


@pytest.mark.parametrize("shape", [RAGGED, RAGGED64, RAGGED64_ODD])
@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_ragged_shapes(shape, prec):
    res = run_steps(shape, prec, 2, 1e-3, 0.9, 0.95, 1e-8, 0.1, "zipf", seed=13,
                    check_grads_every_step=True)
    assert_parity(res, shape, prec)


def test_gpt2_124m_shapes_short_sequence_bf16():
    """Every weight at its full 124M size (all tiles of the 50304-wide head),
    on a batch the oracle can finish in seconds."""
    shape = GPT2_124M + (1, 64)
    res = run_steps(shape, "bf16", 1, 6e-4, 0.9, 0.999, 1e-8, 0.1, "zipf", seed=14)
    assert_parity(res, shape, "bf16")


def _prefix_losses(shape, prec, rows, tprefix, dist, seed):
    """Full-size step on the GPU; the per-position losses of the first
    `tprefix` positions of `rows` rows depend only on those positions (causal
    mask), so the oracle checks them on the truncated batch."""
    L, C, NH, V, Vp, maxT, B, T = shape
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision=prec, seed=seed)
    tok, tgt = synthetic.batch(seed + 1, B, T, V, dist)
    p0 = m.copy_out(PARAMS)
    loss = m.forward(cuda_ids(tok), cuda_ids(tgt))
    got = m.losses().reshape(B, T)[:rows, :tprefix]
    m.zero_grad()
    m.backward()
    g = m.copy_out(GRADS)
    m.adamw_step(6e-4, 0.9, 0.999, 1e-8, 0.1, 1)
    p1 = m.copy_out(PARAMS)
    cfg = oracle.cfg8(L, C, NH, V, Vp, maxT, rows, tprefix)
    ref = oracle.fwdbwd(cfg, p0, tok[:rows, :tprefix], tgt[:rows, :tprefix], want_grads=False)["losses"]
    return loss, got.reshape(-1), ref, g, p0, p1, m


@pytest.mark.parametrize("shape,rows,tp,dist", [
    (GPT2_124M + (4, 1024), 1, 1024, "uniform"),  # 124M, B=4 single step: one whole row
    (GPT2_124M + (16, 1024), 2, 32, "zipf"),      # 124M throughput shape
    ((24, 1024, 16, 50257, 50304, 1024, 8, 1024), 2, 24, "uniform"),  # 350M
])
def test_full_size_sampled(shape, rows, tp, dist):
    L, C, NH, V, Vp, maxT, B, T = shape
    loss, got, ref, g, p0, p1, m = _prefix_losses(shape, "bf16", rows, tp, dist, seed=21)
    np.testing.assert_allclose(got, ref, atol=TOL["bf16"]["loss"] * 3, rtol=0)
    assert abs(float(np.mean(got)) - float(np.mean(ref))) <= TOL["bf16"]["loss"]
    # at init the logits are ~N(0, C * 0.02^2) (unit-variance LN output times
    # std-0.02 embedding rows), so E[loss] ~ ln V + C * 0.02^2 / 2
    assert abs(loss - (math.log(V) + C * 0.02 ** 2 / 2)) < 0.05
    assert np.all(np.isfinite(g))
    # AdamW at t = 1: |m_hat / (sqrt(v_hat) + eps)| <= 1, so every parameter
    # moves by at most lr beyond its decay
    lr, wd = 6e-4, 0.1
    assert np.max(np.abs(p1 - p0 * (1 - lr * wd))) <= lr * (1 + 1e-5) + 1e-7
    tab = dict((n, (o, k)) for n, o, k in m.tensor_table())
    o, k = tab["wte"]
    assert np.all(p1[o + V * C:o + k] == 0)


def test_errors_are_reported():
    L, C, NH, V, Vp, maxT, B, T = TINY
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=1)
    with pytest.raises(GPT2Error) as e:
        m.backward()
    assert e.value.code == -4  # GPT2_ERR_STATE
    with pytest.raises(GPT2Error) as e:
        m.adamw_step(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)
    assert e.value.code == -1
    tok, tgt = synthetic.batch(2, B, T, V)
    bad = tok.copy()
    bad[1, 3] = V + 5
    with pytest.raises(GPT2Error) as e:
        m.forward(cuda_ids(bad), cuda_ids(tgt))
    assert e.value.code == -5  # GPT2_ERR_TOKEN
    badt = tgt.copy()
    badt[0, 0] = -1
    with pytest.raises(GPT2Error) as e:
        m.forward(cuda_ids(tok), cuda_ids(badt))
    assert e.value.code == -5
    # the model stays usable after a reported error
    loss = m.forward(cuda_ids(tok), cuda_ids(tgt))
    assert math.isfinite(loss)
    with pytest.raises(GPT2Error) as e:
        m.residual(L + 1)
    assert e.value.code == -1


def test_host_entry_point_matches_device_entry_point():
    L, C, NH, V, Vp, maxT, B, T = RAGGED
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=5)
    tok, tgt = synthetic.batch(6, B, T, V)
    a = m.forward(cuda_ids(tok), cuda_ids(tgt))
    ht = torch.from_numpy(tok).pin_memory()
    hg = torch.from_numpy(tgt).pin_memory()
    b = m.forward_host(ht, hg)
    assert a == b


def test_step_is_deterministic():
    L, C, NH, V, Vp, maxT, B, T = CHAR
    out = []
    for _ in range(2):
        m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=9)
        tok, tgt = synthetic.batch(10, B, T, V, "zipf")
        m.forward(cuda_ids(tok), cuda_ids(tgt))
        m.zero_grad()
        m.backward()
        out.append(m.copy_out(GRADS))
        m.close()
    assert np.array_equal(out[0], out[1])


def test_stream_is_honoured():
    L, C, NH, V, Vp, maxT, B, T = TINY
    s = torch.cuda.Stream()
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=3, stream=s)
    tok, tgt = synthetic.batch(2, B, T, V)
    with torch.cuda.stream(s):
        t1, t2 = cuda_ids(tok), cuda_ids(tgt)
    loss = m.forward(t1, t2)
    assert math.isfinite(loss)


def test_named_array_copies_and_device_loss_pointer():
    # gpt2_copy_{params,grads,m,v}_out / gpt2_copy_params_in against the
    # arena-indexed copies, and the device mean-loss address against
    # gpt2_read_loss, after one full step
    import ctypes
    from cuda.bindings import runtime as rt
    from transformer_lm_step_gpt_b300 import ADAM_M, ADAM_V, load_library
    L, C, NH, V, Vp, maxT, B, T = TINY
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=31)
    lib = load_library()
    tok, tgt = synthetic.batch(32, B, T, V)
    m.forward(cuda_ids(tok), cuda_ids(tgt))
    m.zero_grad()
    m.backward()
    m.adamw_step(1e-3, 0.9, 0.999, 1e-8, 0.1, 1)
    m.forward(cuda_ids(tok), cuda_ids(tgt), sync=False)
    m.synchronize()
    n = m.num_params
    for fn, arena in [(lib.gpt2_copy_params_out, PARAMS), (lib.gpt2_copy_grads_out, GRADS),
                      (lib.gpt2_copy_m_out, ADAM_M), (lib.gpt2_copy_v_out, ADAM_V)]:
        a = np.empty(n, np.float32)
        assert fn(m._h, a.ctypes.data) == 0
        assert np.array_equal(a, m.copy_out(arena))
    p = np.random.default_rng(3).normal(0, 0.02, n).astype(np.float32)
    assert lib.gpt2_copy_params_in(m._h, p.ctypes.data) == 0
    assert np.array_equal(m.copy_out(PARAMS), p)
    m.forward(cuda_ids(tok), cuda_ids(tgt), sync=False)
    m.synchronize()
    ptr = m.loss_device_ptr()
    assert ptr
    host = np.zeros(1, np.float32)
    (err,) = rt.cudaMemcpy(host.ctypes.data, ptr, 4, rt.cudaMemcpyKind.cudaMemcpyDefault)
    assert err == rt.cudaError_t.cudaSuccess
    assert host[0] == np.float32(m.read_loss())
    assert lib.gpt2_loss_device_ptr(None, None) == -1


def test_expired_wait_is_reported_and_the_model_recovers():
    # a kernel whose bounded mbarrier wait nothing completes: it gives up
    # after the limit, the next synchronising call reports GPT2_ERR_TIMEOUT,
    # and the model keeps working (the same step repeats bit for bit)
    import time
    L, C, NH, V, Vp, maxT, B, T = TINY
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=41)
    tok, tgt = synthetic.batch(42, B, T, V)
    l0 = m.forward(cuda_ids(tok), cuda_ids(tgt))
    t0 = time.time()
    m.expire_a_wait()
    with pytest.raises(GPT2Error) as e:
        m.synchronize()
    assert e.value.code == -6
    assert time.time() - t0 >= 1.5
    m.synchronize()   # the condition was cleared
    assert m.forward(cuda_ids(tok), cuda_ids(tgt)) == l0


# ---- whole-step parity at the configurations' sequence length: every gradient
# ---- tensor, updated parameter, m and v against the oracle on one-layer
# ---- models small enough for the oracle, but on the launch paths the 124M and
# ---- 350M steps take (causal mask: GeekNews, "A GPT-2-based ChatGPT clone in
# ---- 3000 bytes of C", *The Transformer core*; per-layer backward: QbitAI,
# ---- "OpenAI founder hand-writes...", *Manually implementing each layer's
# ---- forward/backward pass*)

# T = 1024, B = 4 (M = 4096): the attention kernels walk 16 key blocks of 64
# and 8 of 128 for the last query rows; the qkv and attproj weight gradients
# have fewer output tiles than SMs and K = 4096, so their split-K runs more
# than 4 ways and is reduced by the separate split-order kernel
LONG1024 = (1, 128, 2, 1000, 1000, 1024, 4, 1024)
# T = 4096, one sequence, head size 64: 64 key blocks of 64 per query row
LONG4096 = (1, 128, 2, 1000, 1000, 4096, 1, 4096)
# C = 1024, 16 heads (the 350M layer): the LayerNorm kernels' widest rows and
# every 350M matmul shape; the attproj weight gradient (4 x 4 tiles of 256 on
# CTA pairs) splits K = 4096 four ways, reduced inside the matmul in split order
WIDE1024 = (1, 1024, 16, 1000, 1000, 1024, 4, 1024)
# C = 256, 4 heads: every weight gradient runs on CTA pairs with one to four
# 256 x 256 tiles, so K = 4096 splits 8 ways into partial planes that the
# split-order kernel adds up (the path of the 124M attproj weight gradient)
MID1024 = (1, 256, 4, 1000, 1000, 1024, 4, 1024)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_long_sequence_whole_step(prec):
    res = run_steps(LONG1024, prec, 2, 1e-3, 0.9, 0.95, 1e-8, 0.1, "zipf", seed=15,
                    check_grads_every_step=True)
    assert_parity(res, LONG1024, prec)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_longest_sequence_whole_step(prec):
    res = run_steps(LONG4096, prec, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1, "uniform", seed=16)
    assert_parity(res, LONG4096, prec)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_widest_layer_whole_step(prec):
    res = run_steps(WIDE1024, prec, 1, 6e-4, 0.9, 0.999, 1e-8, 0.1, "uniform", seed=17)
    assert_parity(res, WIDE1024, prec)


def test_pair_split_planes_whole_step():
    res = run_steps(MID1024, "bf16", 1, 6e-4, 0.9, 0.999, 1e-8, 0.1, "zipf", seed=18)
    assert_parity(res, MID1024, "bf16")


# one layer of the 124M model's width at its throughput batch (B = 16,
# T = 1024): every product of a layer runs at the step's own shapes (192
# tiles of 256 x 256 on the N = 768 products, more than two waves of CTA
# pairs), and every gradient, parameter, m and v is compared
FULLWIDTH = (1, 768, 12, 1000, 1024, 1024, 16, 1024)


def test_full_width_layer_whole_step():
    res = run_steps(FULLWIDTH, "bf16", 1, 6e-4, 0.9, 0.999, 1e-8, 0.1, "zipf", seed=20)
    assert_parity(res, FULLWIDTH, "bf16")


# a vocabulary row of 120,000 logits (240 KB in bf16, 480 KB in fp32) is
# larger than a block's shared memory, so the softmax / cross-entropy takes
# the streaming kernel (two passes over the row in global memory) instead of
# the one that stages the row in shared memory; a row of 114,688 bf16 logits
# is the largest the staged kernel takes (fourteen 16 KB pieces, all full)
BIGVOCAB = (1, 32, 2, 120000, 120000, 8, 2, 8)
EDGEVOCAB = (1, 32, 2, 114680, 114688, 8, 2, 8)


@pytest.mark.parametrize("shape", [BIGVOCAB, EDGEVOCAB])
@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_vocabulary_row_larger_than_shared_memory(shape, prec):
    res = run_steps(shape, prec, 2, 1e-3, 0.9, 0.999, 1e-8, 0.1, "zipf", seed=19,
                    check_grads_every_step=True)
    assert_parity(res, shape, prec)


# ---- the edges of what the build accepts (head sizes 32 and 128, single-token
# ---- sequences, the largest shapes, an allocation that cannot succeed); kept
# ---- last, so that with -x a failure here does not hide the results above

@pytest.mark.parametrize("shape", [RAGGED32, RAGGED128])
@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_ragged_shapes_head_sizes_32_and_128(shape, prec):
    test_ragged_shapes(shape, prec)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_single_token_sequences(prec):
    # T = 1: each position attends only to itself, so the softmax has no
    # gradient and the query and key rows of qkvw and qkvb get an exactly zero
    # gradient in the oracle (rounding-level on the GPU).  The loss and every
    # gradient tensor are compared with the oracle; the parameters that
    # AdamW's first step moves by the sign of that rounding are not.
    L, C, NH, V, Vp, maxT, B, T = SINGLE_TOKEN
    res = run_steps(SINGLE_TOKEN, prec, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1, "zipf", seed=13)
    tol = TOL[prec]
    assert abs(res["loss_gpu"][0] - res["loss_ref"][0]) <= tol["loss"]
    bad = {k: v for k, v in res["grad_err"][0].items() if not v <= tol["rel"]}
    assert not bad, bad
    tab = dict((n, (o, k)) for n, o, k in res["tab"])
    g = res["grads_gpu"]
    o, _ = tab["qkvw"]
    w = g[o:o + 3 * C * C].reshape(3 * C, C)       # rows q | k | v
    assert np.linalg.norm(w[:2 * C]) <= 1e-3 * np.linalg.norm(w[2 * C:])
    o, _ = tab["qkvb"]
    b = g[o:o + 3 * C]
    assert np.linalg.norm(b[:2 * C]) <= 1e-3 * np.linalg.norm(b[2 * C:])


@pytest.mark.parametrize("shape,rows,tp,dist", [
    # the largest shapes the build accepts, one layer each: T = 4096 with
    # B*T = 32768 and C = 1024; and Vp*B*T just below 2^32 (4.29e9 logits,
    # past 2^31: every index into them must be 64-bit)
    ((1, 1024, 16, 50257, 50304, 4096, 8, 4096), 1, 24, "uniform"),
    ((1, 1024, 16, 131064, 131064, 1024, 32, 1024), 1, 16, "uniform"),
])
def test_largest_accepted_shapes_sampled(shape, rows, tp, dist):
    test_full_size_sampled(shape, rows, tp, dist)


def test_out_of_memory_is_reported_and_the_context_stays_usable():
    # 2048 layers of C = 1024 need ~0.5 TB for the parameters and optimizer
    # state alone: the build's one cudaMalloc fails, which is GPT2_ERR_OOM
    with pytest.raises(GPT2Error) as e:
        Model(2048, 1024, 16, 50257, 50304, 1024, 1, 1024, precision="bf16", seed=1)
    assert e.value.code == -2  # GPT2_ERR_OOM
    L, C, NH, V, Vp, maxT, B, T = TINY
    m = Model(L, C, NH, V, Vp, maxT, B, T, precision="bf16", seed=1)
    tok, tgt = synthetic.batch(2, B, T, V)
    assert math.isfinite(m.forward(cuda_ids(tok), cuda_ids(tgt)))
