"""Seeded synthetic inputs: token streams and parameter arrays.

This module feeds both the CUDA library and its CPU oracle the *same* inputs.
It holds none of the method's arithmetic (no layer, no loss, no optimiser):
only random numbers, drawn from documented generators, shaped like the
workloads the method is measured on.

Token stream
    One stream of B*(T+1) ids per batch, drawn with SplitMix64 (Steele, Lea,
    Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
    seeded with ``seed ^ 0x9E3779B97F4A7C15``.  Row b is
    ``s[b*(T+1) : (b+1)*(T+1)]``; tokens = row[:T], targets = row[1:]
    (next-token language modelling).  A 53-bit uniform u in [0,1) picks the
    id: ``floor(u*V)`` for "uniform", or the inverse CDF of Zipf(s=1.1) over
    [0, V) with P(k) proportional to (k+1)^-1.1 (rank = id) for "zipf", a
    natural-text rank-frequency stand-in for the public corpora the method
    was trained on (none of which is used here).

Parameters
    ``gpt2_init``: N(0, 0.02) for the embedding and Linear weights, the two
    residual projections scaled by 1/sqrt(2L), biases 0, LayerNorm gamma 1
    and beta 0, vocabulary pad rows 0 -- drawn with numpy's PCG64.
    ``perturbed``: the same plus N(0, 0.02) biases and LayerNorm gamma/beta
    offsets, so that parity tests exercise every term.
    The caller supplies the tensor table (name, offset, numel) of the 1-D
    parameter array; nothing here knows the model's layout.
"""
import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """First n outputs of SplitMix64 started at state ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform53(seed: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from the top 53 bits of SplitMix64."""
    x = splitmix64(seed, n) >> np.uint64(11)
    return x.astype(np.float64) * (1.0 / 9007199254740992.0)


def zipf_cdf(V: int, s: float = 1.1) -> np.ndarray:
    w = (np.arange(V, dtype=np.float64) + 1.0) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def token_stream(seed: int, n: int, V: int, dist: str = "uniform") -> np.ndarray:
    u = uniform53(seed ^ 0x9E3779B97F4A7C15, n)
    if dist == "uniform":
        ids = np.floor(u * V).astype(np.int64)
    elif dist == "zipf":
        ids = np.searchsorted(zipf_cdf(V), u, side="right")
    else:
        raise ValueError(dist)
    return np.minimum(ids, V - 1).astype(np.int32)


def batch(seed: int, B: int, T: int, V: int, dist: str = "uniform"):
    """(tokens [B,T], targets [B,T]) int32, next-token pairs from one stream."""
    s = token_stream(seed, B * (T + 1), V, dist).reshape(B, T + 1)
    return np.ascontiguousarray(s[:, :T]), np.ascontiguousarray(s[:, 1:])


_NORMAL_W = {"wte", "wpe", "qkvw", "fcw"}
_RESID_W = {"attprojw", "fcprojw"}
_GAMMA = {"ln1w", "ln2w", "lnfw"}


def params(table, L: int, C: int, V: int, seed: int, kind: str = "gpt2_init",
           dtype=np.float32) -> np.ndarray:
    """Parameter array for the given tensor table [(name, offset, numel)]."""
    total = max(off + n for _, off, n in table)
    p = np.zeros(total, np.float64)
    rng = np.random.Generator(np.random.PCG64(seed))
    sd, sdr = 0.02, 0.02 / np.sqrt(2.0 * max(L, 1))
    for name, off, n in table:
        if name in _NORMAL_W:
            v = rng.normal(0.0, sd, n)
            if name == "wte":
                v[V * C:] = 0.0  # pad rows stay zero
        elif name in _RESID_W:
            v = rng.normal(0.0, sdr, n)
        elif name in _GAMMA:
            v = np.ones(n)
            if kind == "perturbed":
                v += rng.normal(0.0, 0.1, n)
        else:  # biases, LayerNorm beta
            v = np.zeros(n)
            if kind == "perturbed":
                v += rng.normal(0.0, 0.02, n)
        p[off:off + n] = v
    return p.astype(dtype)
