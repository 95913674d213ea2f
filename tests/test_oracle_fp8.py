"""Pins of the oracle's FP8 (E4M3) format and scaled matmul (CPU only).

E4M3 is fixed by its definition (OCP 8-bit floating point: 1 sign, 4
exponent bits with bias 7, 3 mantissa bits, subnormals at exponent 0,
S.1111.111 = NaN, no infinity, largest finite 448); the pins check the
oracle's decoder against values written out from that definition, its
encoder against a brute-force nearest-code search done here with numpy,
and the tie and saturation rules at chosen points.
"""
import math

import numpy as np
import pytest

import oracle


def test_decode_closed_forms():
    want = {
        0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
        0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0,
    }
    for c, v in want.items():
        assert oracle.e4m3_decode(c) == v, hex(c)
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_codes_increase_and_round_trip():
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def nearest_code(x):
    """Brute force: the code of least |x - value| among the finite codes of
    x's sign, ties to the even mantissa field, magnitudes over 448 -> 448."""
    codes = np.arange(0x7F)
    vals = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    a = min(abs(x), 448.0)
    d = np.abs(vals - a)
    best = np.flatnonzero(d == d.min())
    c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (0x80 if math.copysign(1.0, x) < 0 else 0)


def test_encode_matches_brute_force():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.normal(0, 1, 300), rng.normal(0, 100, 200), rng.uniform(-1e-2, 1e-2, 200),
                         rng.uniform(-600, 600, 100)])
    for x in xs:
        assert oracle.e4m3_encode(float(x)) == nearest_code(float(x)), x


def test_ties_and_saturation():
    assert oracle.e4m3_encode(1.0625) == 0x38      # halfway 1.0 | 1.125 -> even mantissa (1.0)
    assert oracle.e4m3_encode(1.1875) == 0x3A      # halfway 1.125 | 1.25 -> 1.25
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal -> 0
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02
    assert oracle.e4m3_encode(-3 * 2.0 ** -10) == 0x82
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E and oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_quantize_per_tensor_scale():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (7, 33)).astype(np.float32)
    x[3, 5] = -12.5   # the largest magnitude
    q, s = oracle.fp8_quantize(x)
    assert s == np.float32(448.0) / np.float32(12.5)
    assert q[3, 5] == 0xFE
    for (i, j) in [(0, 0), (6, 32), (2, 17)]:
        assert q[i, j] == oracle.e4m3_encode(float(np.float32(x[i, j]) * np.float32(s)))
    z, s0 = oracle.fp8_quantize(np.zeros((4, 4), np.float32))
    assert s0 == 1.0 and not z.any()


def test_fp8_matmul_selects_and_scales():
    # B rows are one-hot 1.0 codes: out[m, n] picks column perm[n] of A
    rng = np.random.default_rng(2)
    M, N, K = 5, 4, 16
    qa = rng.integers(0, 0x7F, (M, K)).astype(np.uint8)
    qa[qa == 0x7F] = 0x38
    perm = [3, 0, 15, 7]
    qb = np.zeros((N, K), np.uint8)
    for n, k in enumerate(perm):
        qb[n, k] = 0x38
    out = oracle.fp8_matmul(qa, 2.0, qb, 4.0, bias=[1.0, 2.0, 3.0, 4.0])
    for m in range(M):
        for n, k in enumerate(perm):
            assert out[m, n] == oracle.e4m3_decode(int(qa[m, k])) / 8.0 + (n + 1)
