"""Seeded synthetic inputs: token streams and initial weights.

This module draws random numbers and nothing else. It holds none of the model's
arithmetic, so both the CPU oracle's tests and the GPU path can take their inputs
from it.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used in counter mode so that any element of any stream
can be drawn directly:

    mix(z)      = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
                  z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)
    draw(k, i)  = mix(k + (i + 1) * 0x9E3779B97F4A7C15)          (mod 2**64)
    key(s, j)   = draw(s, j)              (stream j of seed s)
    uniform     = (draw >> 11) * 2**-53   in [0, 1)
    normal pair = Box-Muller on uniforms (2n, 2n+1):
                  r = sqrt(-2 ln(1 - u0)),  (r cos(2 pi u1), r sin(2 pi u1))

The library's own initialiser (gpt2_create) implements the same definition in C++;
a CPU test checks that the two agree.

Workload recipe (the pages train on OpenWebText and Shakespeare text, neither of
which is available, so seeded ids of the same shape stand in for them):
  * tokens: a stream of T+1 ids per row; inputs are ids[:, :T], targets ids[:, 1:]
    (the next-token shift of 「从零实现一个最小GPT」 二.2, get_batch).
  * ids are uniform over [0, V) or Zipf(s) with P(i) proportional to (i+1)**-s,
    sampled by inverse CDF (lowest i whose CDF >= u).
  * weights: N(0, 0.02) for embeddings and Linear weights (「从零实现一个最小GPT」 三.7,
    "_init_weights"), the two residual projections scaled by 1/sqrt(2 L),
    Linear biases 0, LayerNorm gamma 1 and beta 0, padded vocabulary rows 0.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def draw(key: int, index: np.ndarray) -> np.ndarray:
    """64-bit outputs number `index` (array) of the stream with key `key`."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * _GOLDEN
    return _mix(z)


def stream_key(seed: int, stream: int) -> int:
    return int(draw(seed & 0xFFFFFFFFFFFFFFFF, np.array([stream], dtype=np.uint64))[0])


def uniform(key: int, n: int, start: int = 0) -> np.ndarray:
    """n doubles in [0, 1) from positions start..start+n-1 of the stream."""
    bits = draw(key, np.arange(start, start + n, dtype=np.uint64))
    return (bits >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller pairs over consecutive uniforms)."""
    pairs = (n + 1) // 2
    u = uniform(key, 2 * pairs)
    u0, u1 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u0))
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u1)
    out[1::2] = r * np.sin(2.0 * np.pi * u1)
    return out[:n]


def zipf_cdf(vocab: int, s: float) -> np.ndarray:
    w = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
    return np.cumsum(w) / w.sum()


def token_stream(seed: int, batch_index: int, B: int, T: int, vocab: int,
                 dist: str = "uniform", s: float = 1.0) -> np.ndarray:
    """int32 [B, T+1] ids for batch number `batch_index` of seed `seed`."""
    key = stream_key(seed, 1_000_000 + batch_index)
    u = uniform(key, B * (T + 1))
    if dist == "uniform":
        ids = np.minimum((u * vocab).astype(np.int64), vocab - 1)
    elif dist == "zipf":
        cdf = zipf_cdf(vocab, s)
        ids = np.minimum(np.searchsorted(cdf, u, side="left"), vocab - 1)
    else:
        raise ValueError(dist)
    return ids.reshape(B, T + 1).astype(np.int32)


def batch(seed: int, batch_index: int, B: int, T: int, vocab: int,
          dist: str = "uniform", s: float = 1.0):
    """(tokens, targets), both int32 [B, T]; targets are tokens shifted by one."""
    ids = token_stream(seed, batch_index, B, T, vocab, dist, s)
    return np.ascontiguousarray(ids[:, :T]), np.ascontiguousarray(ids[:, 1:])


# Parameter table shared by the ABI and the tests: (name, shape builder, init kind).
# init kind: "w" N(0, 0.02); "wres" N(0, 0.02/sqrt(2L)); "zero"; "one".
_TABLE = [
    ("wte", lambda c: (c["Vp"], c["C"]), "w"),
    ("wpe", lambda c: (c["T"], c["C"]), "w"),
    ("ln1w", lambda c: (c["L"], c["C"]), "one"),
    ("ln1b", lambda c: (c["L"], c["C"]), "zero"),
    ("qkvw", lambda c: (c["L"], 3 * c["C"], c["C"]), "w"),
    ("qkvb", lambda c: (c["L"], 3 * c["C"]), "zero"),
    ("attprojw", lambda c: (c["L"], c["C"], c["C"]), "wres"),
    ("attprojb", lambda c: (c["L"], c["C"]), "zero"),
    ("ln2w", lambda c: (c["L"], c["C"]), "one"),
    ("ln2b", lambda c: (c["L"], c["C"]), "zero"),
    ("fcw", lambda c: (c["L"], 4 * c["C"], c["C"]), "w"),
    ("fcb", lambda c: (c["L"], 4 * c["C"]), "zero"),
    ("fcprojw", lambda c: (c["L"], c["C"], 4 * c["C"]), "wres"),
    ("fcprojb", lambda c: (c["L"], c["C"]), "zero"),
    ("lnfw", lambda c: (c["C"],), "one"),
    ("lnfb", lambda c: (c["C"],), "zero"),
]
BIAS_NAMES = ("qkvb", "attprojb", "fcb", "fcprojb")


def param_table(V: int, Vp: int, T: int, L: int, C: int, bias: bool):
    """[(stream index, name, shape, init kind)] in buffer order; stream index is the
    row of the full table, so it does not change when biases are absent."""
    c = dict(V=V, Vp=Vp, T=T, L=L, C=C)
    out = []
    for i, (name, shape, kind) in enumerate(_TABLE):
        if not bias and name in BIAS_NAMES:
            continue
        out.append((i, name, tuple(shape(c)), kind))
    return out


def init_params(seed: int, V: int, Vp: int, T: int, L: int, C: int, bias: bool,
                dtype=np.float32) -> dict:
    """Initial weights as a dict name -> array (fp32 by default)."""
    params = {}
    for stream, name, shape, kind in param_table(V, Vp, T, L, C, bias):
        n = int(np.prod(shape))
        if kind == "zero":
            a = np.zeros(n)
        elif kind == "one":
            a = np.ones(n)
        else:
            std = 0.02 if kind == "w" else 0.02 / np.sqrt(2.0 * L)
            a = np.zeros(n)
            real = V * C if name == "wte" else n   # padded vocabulary rows stay 0
            a[:real] = std * normal(stream_key(seed, stream), real)
        params[name] = a.reshape(shape).astype(dtype)
    return params


# The workloads, by name: shapes, token distribution and seeds.
WORKLOADS = {
    "tiny-fp32": dict(V=65, Vp=128, T=64, L=4, H=4, C=128, bias=False, B=4, accum=1,
                      precision="fp32", dist="uniform", s=0.0, tok_seed=0, w_seed=1000),
    "char-bf16": dict(V=65, Vp=128, T=256, L=6, H=6, C=384, bias=True, B=64, accum=1,
                      precision="bf16", dist="zipf", s=1.1, tok_seed=1, w_seed=1001),
    "gpt2-124m-micro": dict(V=50257, Vp=50304, T=1024, L=12, H=12, C=768, bias=True, B=12,
                            accum=1, precision="bf16", dist="zipf", s=1.0, tok_seed=2,
                            w_seed=1002),
    "gpt2-124m-step": dict(V=50257, Vp=50304, T=1024, L=12, H=12, C=768, bias=True, B=12,
                           accum=40, precision="bf16", dist="zipf", s=1.0, tok_seed=2,
                           w_seed=1003),
    "gpt2-350m-shape": dict(V=50257, Vp=50304, T=1024, L=24, H=16, C=1024, bias=True, B=8,
                            accum=8, precision="bf16", dist="zipf", s=1.0, tok_seed=2,
                            w_seed=1004),
}
