"""Seeded synthetic inputs shared by the CUDA path's drivers and by the oracle.

This module draws numbers and builds token sequences. It holds none of the
attention or cache arithmetic: it never matches, allocates, evicts or attends.

Everything is keyed on SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used here as a counter-based
mixing function:

    mix64(x) = finalizer(x + 0x9E3779B97F4A7C15)
    finalizer(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
                  z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31

(all arithmetic mod 2**64). mix64(0), mix64(GOLDEN), ... reproduce the
published SplitMix64 stream for seed 0.

Synthetic model. The KV of a token depends only on the tokens before it and
the token itself (the pages' observation that KV is a function of the prefix),
so every Q/K/V row is keyed on a rolling prefix hash:

    h[-1] = seed;  h[j] = mix64(h[j-1] ^ (t[j] + GOLDEN))

and a row of `head_dim` values for (tensor, layer, head) is

    key  = mix64((tensor << 48) | (layer << 24) | head)      tensor: Q=1, K=2, V=3
    base = mix64(h[j] ^ key)
    u_e  = mix64(base + e)                                    e = 0 .. head_dim-1
    s_e  = sum of the four 16-bit fields of u_e               (0 .. 262140)
    x_e  = float32(s_e - 131070) * float32(sqrt(3) / 65536)   (one fp32 multiply, RNE)

i.e. an Irwin-Hall(4) approximation of N(0, 1) (mean 0, variance 1 - 2**-32,
bounded by +-3.4641). bf16 values are the round-to-nearest-even bf16 of x_e.
Integer work plus one IEEE multiply: host and device produce identical bits.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
VALUE_SCALE = np.float32(np.sqrt(3.0) / 65536.0)
TENSOR_Q, TENSOR_K, TENSOR_V = 1, 2, 3
VOCAB = 32000

_U64 = np.uint64


def mix64(x):
    """SplitMix64 output for state `x` (array or scalar, uint64, wrapping)."""
    with np.errstate(over="ignore"):
        z = np.asarray(x, dtype=np.uint64) + GOLDEN
        z = (z ^ (z >> _U64(30))) * _M1
        z = (z ^ (z >> _U64(27))) * _M2
        return z ^ (z >> _U64(31))


def stream(seed: int, stream_id: int, n: int, start: int = 0) -> np.ndarray:
    """n uint64 draws of the counter stream (seed, stream_id): mix64(key + i)."""
    key = mix64(_U64(seed) ^ mix64(_U64(stream_id)))
    with np.errstate(over="ignore"):
        return mix64(key + np.arange(start, start + n, dtype=np.uint64))


def tokens(seed: int, stream_id: int, n: int, start: int = 0) -> np.ndarray:
    """n token ids uniform in [0, VOCAB) (draw mod VOCAB), int32."""
    return (stream(seed, stream_id, n, start) % _U64(VOCAB)).astype(np.int32)


def prefix_hashes(seed: int, toks: np.ndarray, h0=None) -> np.ndarray:
    """Rolling prefix hash h[j] for every position of one token sequence.

    `h0` continues a chain (the hash of the token before toks[0]); default `seed`.
    """
    toks = np.asarray(toks, dtype=np.int64).astype(np.uint64)
    out = np.empty(len(toks), dtype=np.uint64)
    h = _U64(seed) if h0 is None else _U64(h0)
    with np.errstate(over="ignore"):
        add = toks + GOLDEN
        for j in range(len(toks)):
            h = mix64(h ^ add[j])
            out[j] = h
    return out


def prefix_hashes_batch(seed: int, seqs) -> list:
    """prefix_hashes for many sequences, vectorised across sequences."""
    seqs = [np.asarray(s, dtype=np.int64) for s in seqs]
    if not seqs:
        return []
    n = len(seqs)
    lens = np.array([len(s) for s in seqs], dtype=np.int64)
    maxlen = int(lens.max()) if n else 0
    pad = np.zeros((n, maxlen), dtype=np.uint64)
    for i, s in enumerate(seqs):
        pad[i, : len(s)] = s.astype(np.uint64)
    out = np.empty((n, maxlen), dtype=np.uint64)
    h = np.full(n, seed, dtype=np.uint64)
    with np.errstate(over="ignore"):
        add = pad + GOLDEN
        for j in range(maxlen):
            h = mix64(h ^ add[:, j])
            out[:, j] = h
    return [out[i, : lens[i]].copy() for i in range(n)]


def stream_key(tensor: int, layer: int, head: int) -> np.uint64:
    return mix64(_U64((tensor << 48) | (layer << 24) | head))


def _fields_sum(u: np.ndarray) -> np.ndarray:
    m = _U64(0xFFFF)
    return ((u & m) + ((u >> _U64(16)) & m) + ((u >> _U64(32)) & m) + (u >> _U64(48))).astype(np.int64)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (uint16). Finite inputs only."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def values_f32(hashes: np.ndarray, tensor: int, layer: int, heads, head_dim: int) -> np.ndarray:
    """float32 values [n, len(heads), head_dim] for the given prefix hashes (fp32 model)."""
    hashes = np.asarray(hashes, dtype=np.uint64)
    heads = list(heads)
    out = np.empty((len(hashes), len(heads), head_dim), dtype=np.float32)
    e = np.arange(head_dim, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for hi, h in enumerate(heads):
            base = mix64(hashes ^ stream_key(tensor, layer, h))
            u = mix64(base[:, None] + e[None, :])
            s = _fields_sum(u) - 131070
            out[:, hi, :] = s.astype(np.float32) * VALUE_SCALE
    return out


def values(hashes, tensor: int, layer: int, heads, head_dim: int, dtype: str) -> np.ndarray:
    """Values in the model dtype, returned as float32 (bf16-rounded when dtype == 'bf16')."""
    v = values_f32(hashes, tensor, layer, heads, head_dim)
    if dtype == "bf16":
        return bf16_bits_to_f32(to_bf16_bits(v))
    if dtype == "f32":
        return v
    raise ValueError(dtype)


def values_bits(hashes, tensor: int, layer: int, heads, head_dim: int, dtype: str) -> np.ndarray:
    """Storage bits of the values: uint16 for bf16, float32 for f32."""
    v = values_f32(hashes, tensor, layer, heads, head_dim)
    return to_bf16_bits(v) if dtype == "bf16" else v


def permutation(seed: int, n: int, stream_id: int = 0x5045524D) -> np.ndarray:
    """Seeded Fisher-Yates permutation of 0..n-1 (int32): for i = n-1..1, j = draw_i mod (i+1)."""
    a = np.arange(n, dtype=np.int32)
    if n <= 1:
        return a
    draws = stream(seed, stream_id, n - 1)
    js = (draws % np.arange(n, 1, -1, dtype=np.uint64)).astype(np.int64)
    for k, i in enumerate(range(n - 1, 0, -1)):
        j = js[k]
        a[i], a[j] = a[j], a[i]
    return a


def irwin_hall_normal(seed: int, stream_id: int, n: int) -> np.ndarray:
    """n approximately N(0,1) draws (float64), Irwin-Hall(4) of 16-bit fields."""
    s = _fields_sum(stream(seed, stream_id, n)) - 131070
    return s.astype(np.float64) * (np.sqrt(3.0) / 65536.0)


def uniform_int(seed: int, stream_id: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (draw mod span)."""
    span = np.uint64(hi - lo + 1)
    return (stream(seed, stream_id, n) % span).astype(np.int64) + lo
