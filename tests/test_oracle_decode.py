"""Pins of the oracle's generation path (CPU only).

The incremental forward with a key/value cache (GeekNews, "A GPT-2-based
ChatGPT clone in 3000 bytes of C", section "How KV caching works") must give,
row by row, the logits of the full causal forward over the same tokens (a
different code path: materialised T x T attention over the whole batch).
The sampling rule (inverse CDF of the softmax at a temperature; greedy at
temperature 0) is pinned by distributions whose CDF is known in closed form.
"""
import math

import numpy as np
import pytest

import oracle

SHAPES = [
    (2, 32, 4, 50, 56, 16, 3, 9),   # several heads, ragged vocabulary padding
    (1, 16, 1, 11, 16, 8, 2, 8),    # one head, T = maxT
    (3, 64, 4, 37, 40, 12, 1, 5),   # head size 16
]


@pytest.mark.parametrize("shape", SHAPES)
def test_incremental_logits_equal_full_forward(shape):
    cfg = oracle.cfg8(*shape)
    L, C, NH, V, Vp, maxT, B, T = shape
    p = oracle.init_params(cfg, 11)
    # larger weights than the init, so that attention is far from uniform
    p = p * 4.0
    rng = np.random.default_rng(3)
    tok = rng.integers(0, V, (B, T)).astype(np.int32)
    full = oracle.fwdbwd(cfg, p, tok, want_grads=False, want_logits=True)["logits"].reshape(B, T, V)
    inc = oracle.decode_logits(cfg, p, tok)
    assert np.abs(full).max() > 0.1
    # the same arithmetic in the same order, row by row: equal to the last bit
    assert np.array_equal(full, inc)


def test_incremental_detects_a_wrong_position():
    # the position embedding must be the one of each row: feeding the same
    # token at every position gives different logits per position
    shape = (1, 16, 2, 9, 16, 8, 1, 6)
    cfg = oracle.cfg8(*shape)
    p = oracle.init_params(cfg, 5) * 4.0
    tok = np.full((1, 6), 3, np.int32)
    inc = oracle.decode_logits(cfg, p, tok)
    assert np.abs(inc[0, 0] - inc[0, 5]).max() > 1e-6


def test_generate_feeds_drawn_tokens_back():
    shape = (2, 32, 4, 50, 56, 16, 3, 16)
    cfg = oracle.cfg8(*shape)
    L, C, NH, V, Vp, maxT, B, T = shape
    p = oracle.init_params(cfg, 2) * 4.0
    rng = np.random.default_rng(9)
    T0, n_new = 5, 7
    prompt = rng.integers(0, V, (B, T0)).astype(np.int32)
    u = rng.random((n_new, B))
    toks, lg = oracle.generate(cfg, p, prompt, n_new, 0.8, u)
    assert np.array_equal(toks[:, :T0], prompt)
    # the scores of new token i are the logits of row T0 - 1 + i of the full
    # sequence (prompt followed by the drawn tokens)
    cfg2 = oracle.cfg8(L, C, NH, V, Vp, maxT, B, T0 + n_new - 1)
    full = oracle.decode_logits(cfg2, p, toks[:, :T0 + n_new - 1])
    for i in range(n_new):
        assert np.array_equal(lg[i], full[:, T0 - 1 + i])
        for b in range(B):
            assert toks[b, T0 + i] == oracle.sample(lg[i, b], 0.8, u[i, b])


def test_generate_up_to_the_last_cache_row():
    shape = (1, 16, 2, 9, 16, 8, 2, 8)
    cfg = oracle.cfg8(*shape)
    p = oracle.init_params(cfg, 4) * 4.0
    prompt = np.array([[1], [2]], np.int32)
    toks, lg = oracle.generate(cfg, p, prompt, 8, 0.0, np.zeros((8, 2)))
    assert toks.shape == (2, 9)
    assert ((toks >= 0) & (toks < 9)).all()


def test_sample_inverse_cdf_closed_form():
    # p = (1, 2, 3) / 6: CDF 1/6, 1/2, 1
    lg = [0.0, math.log(2.0), math.log(3.0)]
    for u, want in [(0.0, 0), (0.1, 0), (0.166, 0), (0.167, 1), (0.49, 1), (0.501, 2), (0.999, 2)]:
        assert oracle.sample(lg, 1.0, u) == want, u
    # temperature 2: p proportional to sqrt(1), sqrt(2), sqrt(3)
    s = 1 + math.sqrt(2) + math.sqrt(3)
    c0, c1 = 1 / s, (1 + math.sqrt(2)) / s
    for u, want in [(c0 - 1e-6, 0), (c0 + 1e-6, 1), (c1 - 1e-6, 1), (c1 + 1e-6, 2)]:
        assert oracle.sample(lg, 2.0, u) == want, u
    # a shift of every score changes nothing
    assert oracle.sample([x + 100.0 for x in lg], 1.0, 0.3) == 1


def test_sample_greedy_and_limits():
    # temperature 0: the first index of the largest score
    assert oracle.sample([1.0, 3.0, 3.0, 0.0], 0.0, 0.7) == 1
    assert oracle.sample([5.0], 0.0, 0.5) == 0
    # a tiny temperature splits the two tied maxima by u
    assert oracle.sample([1.0, 3.0, 3.0, 0.0], 1e-6, 0.25) == 1
    assert oracle.sample([1.0, 3.0, 3.0, 0.0], 1e-6, 0.75) == 2
    # an entry whose probability underflows to 0 is never drawn
    assert oracle.sample([-1000.0, 0.0], 1.0, 0.0) == 1
    # u at the top end falls on the last index with nonzero probability
    assert oracle.sample([0.0, 0.0, -1000.0], 1.0, 1.0) == 1


def test_sample_frequencies_match_the_softmax():
    rng = np.random.default_rng(1)
    lg = rng.normal(size=6)
    p = np.exp(lg - lg.max())
    p /= p.sum()
    u = (np.arange(6000) + 0.5) / 6000  # a stratified grid: exact frequencies
    counts = np.bincount([oracle.sample(lg, 1.0, x) for x in u], minlength=6)
    assert np.abs(counts / 6000 - p).max() < 1.5 / 6000
