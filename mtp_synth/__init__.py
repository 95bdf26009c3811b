"""Seeded synthetic inputs for the MTP draft-layer forward.

This module is shared by the CPU oracle, the CUDA path's tests and the
benchmark.  It only draws numbers and lays them out in the storage formats the
draft layer consumes; it holds none of the layer's arithmetic.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the constants of Vigna's public-domain
``splitmix64.c``), used as a counter-based stream: output ``i`` of the stream
keyed ``key`` is ``mix(key + (i + 1) * GOLDEN)``.  Every tensor has its own
key, derived from the seed and the tensor's name with FNV-1a, so any slice of
any tensor can be regenerated without producing the rest.  Normals come from
the Box-Muller transform over consecutive output pairs.

Value distributions follow the workloads the draft layer is measured on:
4-bit codes uniform in 0..15 packed eight per uint32 with the low nibble
first, per-group scales ``|N(0, 0.02)| / 8``, biases ``-8 * scale + N(0,
1e-3)``, RMSNorm weights ``1 + N(0, 0.1)``, activations, embedding rows and
KV-cache rows ``N(0, 1)``, sink logits ``N(0, 1)``, router weights
``N(0, 0.02)``, tokens uniform in ``[0, vocab)``.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import CONFIGS, LayerConfig, layer_config  # noqa: F401

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for byte in text.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, name: str) -> int:
    """Key of the stream for tensor ``name`` under ``seed``."""
    z = np.array([(seed * 0x9E3779B97F4A7C15 ^ _fnv1a64(name)) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    with np.errstate(over="ignore"):
        return int(_mix(z)[0])


def stream_u64(seed: int, name: str, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start + count - 1`` of the stream for ``name``."""
    key = np.uint64(stream_key(seed, name))
    out = np.empty(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix(key + idx * GOLDEN)
    return out


def uniform01(seed: int, name: str, count: int, start: int = 0) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits of each output."""
    return (stream_u64(seed, name, start, count) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normal(seed: int, name: str, count: int, start: int = 0) -> np.ndarray:
    """Standard normals (float64); element ``i`` depends only on outputs of its Box-Muller pair."""
    p0 = start // 2
    p1 = (start + count + 1) // 2
    out = np.empty(2 * (p1 - p0), dtype=np.float64)

    def fill(lo: int) -> None:
        hi = min(p1, lo + _CHUNK)
        raw = stream_u64(seed, name, 2 * lo, 2 * (hi - lo)) >> np.uint64(11)
        u1 = (raw[0::2].astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
        u2 = raw[1::2].astype(np.float64) * 2.0 ** -53
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        seg = out[2 * (lo - p0): 2 * (hi - p0)]
        seg[0::2] = r * np.cos(t)
        seg[1::2] = r * np.sin(t)

    starts = list(range(p0, p1, _CHUNK))
    if len(starts) > 2:
        # numpy releases the GIL inside these array operations: chunks run in parallel
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    else:
        for lo in starts:
            fill(lo)
    off = start - 2 * p0
    return out[off: off + count]


def normal_f32(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return (mean + std * normal(seed, name, n)).astype(np.float32).reshape(shape)


def norm_weight(seed: int, name: str, dim: int) -> np.ndarray:
    """RMSNorm weight ``1 + N(0, 0.1)``."""
    return normal_f32(seed, name, (dim,), 1.0, 0.1)


def tokens(seed: int, name: str, count: int, vocab: int) -> np.ndarray:
    raw = stream_u64(seed, name, 0, count)
    return (raw % np.uint64(vocab)).astype(np.int32)


def affine4_weight(seed: int, name: str, n: int, k: int):
    """An (N, K) affine 4-bit group-32 weight in storage form.

    Returns ``(q, s, b)``: ``q`` uint32 ``[N, K/8]`` (eight uniform codes per
    word, the code of column ``8*j + i`` in bits ``4*i .. 4*i+3`` of word
    ``j``), ``s`` and ``b`` float32 ``[N, K/32]``.
    """
    if k % 32:
        raise ValueError("K must be a multiple of 32")
    words = n * (k // 8)
    q = (stream_u64(seed, name + ".q", 0, words) >> np.uint64(32)).astype(np.uint32)
    groups = n * (k // 32)
    s = (np.abs(0.02 * normal(seed, name + ".s", groups)) / 8.0).astype(np.float32)
    b = (-8.0 * s.astype(np.float64) + 1e-3 * normal(seed, name + ".b", groups)).astype(np.float32)
    return q.reshape(n, k // 8), s.reshape(n, k // 32), b.reshape(n, k // 32)


def embedding_rows(seed: int, name: str, vocab: int, hidden: int, rows=None) -> np.ndarray:
    """Rows of the float32 ``[vocab, hidden]`` embedding table (all rows when ``rows`` is None)."""
    if rows is None:
        return normal_f32(seed, name, (vocab, hidden))
    out = np.empty((len(rows), hidden), dtype=np.float32)
    for i, r in enumerate(rows):
        if not 0 <= int(r) < vocab:
            raise ValueError("token out of range")
        out[i] = normal(seed, name, hidden, start=int(r) * hidden).astype(np.float32)
    return out


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack integer codes ``[N, K]`` (0..15) into uint32 ``[N, K/8]``, low nibble first.

    Storage-format helper for fixtures that are written as explicit codes.
    """
    codes = np.asarray(codes, dtype=np.uint32)
    n, k = codes.shape
    if k % 8:
        raise ValueError("K must be a multiple of 8")
    if codes.max(initial=0) > 15:
        raise ValueError("codes must be 4-bit")
    c = codes.reshape(n, k // 8, 8)
    word = np.zeros((n, k // 8), dtype=np.uint32)
    for i in range(8):
        word |= c[:, :, i] << np.uint32(4 * i)
    return word
