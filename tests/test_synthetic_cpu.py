"""The seeded input generators both sides share (transformer_lm_step_gpt_b300.synthetic):
SplitMix64 against its published known answers, the uniforms, the Zipf
inverse CDF, the next-token pairing of a batch and reproducibility.  CPU only."""
import os

import numpy as np

from transformer_lm_step_gpt_b300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_known_answers():
    with open(os.path.join(GOLDEN, "splitmix64_kat.txt")) as f:
        want = [int(l, 16) for l in f if l.strip() and not l.startswith("#")]
    got = [int(x) for x in synthetic.splitmix64(0, len(want))]
    assert got == want


def test_uniforms_are_the_top_53_bits():
    u = synthetic.uniform53(0, 3)
    want = [(x >> 11) / 2.0 ** 53 for x in (int(v) for v in synthetic.splitmix64(0, 3))]
    assert list(u) == want
    v = synthetic.uniform53(12345, 100000)
    assert v.min() >= 0.0 and v.max() < 1.0 and abs(v.mean() - 0.5) < 0.005


def test_zipf_cdf_closed_form():
    V, s = 7, 1.1
    w = np.array([(k + 1.0) ** -s for k in range(V)])
    np.testing.assert_allclose(synthetic.zipf_cdf(V, s), np.cumsum(w) / w.sum(), rtol=1e-15)
    assert synthetic.zipf_cdf(V, s)[-1] == 1.0


def test_zipf_stream_frequencies():
    V, n = 50, 200000
    ids = synthetic.token_stream(3, n, V, "zipf")
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < V
    p = np.array([(k + 1.0) ** -1.1 for k in range(V)])
    p /= p.sum()
    f = np.bincount(ids, minlength=V) / n
    # the first ranks hold most of the mass: each within 5 standard errors
    for k in range(5):
        assert abs(f[k] - p[k]) <= 5 * np.sqrt(p[k] * (1 - p[k]) / n), k


def test_batch_is_next_token_pairs_of_one_stream():
    B, T, V = 3, 10, 97
    tok, tgt = synthetic.batch(9, B, T, V, "uniform")
    s = synthetic.token_stream(9, B * (T + 1), V, "uniform").reshape(B, T + 1)
    assert tok.dtype == np.int32 and tok.flags["C_CONTIGUOUS"] and tgt.flags["C_CONTIGUOUS"]
    np.testing.assert_array_equal(tok, s[:, :T])
    np.testing.assert_array_equal(tgt, s[:, 1:])
    np.testing.assert_array_equal(tok[:, 1:], tgt[:, :-1])
    t2, _ = synthetic.batch(9, B, T, V, "uniform")
    np.testing.assert_array_equal(tok, t2)
    t3, _ = synthetic.batch(10, B, T, V, "uniform")
    assert not np.array_equal(tok, t3)
