"""Counter-based random numbers and bf16 rounding for the synthetic workloads.

Generator: the SplitMix64 stream (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Output j of a stream with
seed ``key`` is ``mix64(key + (j + 1) * GOLDEN)``, so any element of any
tensor can be produced on its own.  Every tensor has its own stream:
``key = mix64(mix64(seed) ^ (tensor_id * TID_MULT))``.

* uniform(0,1): ``(h >> 11) * 2**-53`` of output j = flat index.
* standard normal: Box–Muller, cosine branch, from outputs ``2i`` and
  ``2i + 1``: ``sqrt(-2 ln u1) cos(2 pi u2)`` with ``u1`` in (0, 1].

bf16 rounding: float64 -> float32 (numpy, round-to-nearest-even) -> bf16
(round-to-nearest-even on the float32 bit pattern).
"""

from __future__ import annotations

import numpy as np

SEED_BASE = 20261202

# tensor ids inside one workload's stream family
TID = {
    "q": 1, "k": 2, "v": 3, "mix": 4, "x": 5, "w": 6,
    "prefix_k": 7, "prefix_v": 8,
    "step_q": 100, "step_k": 101, "step_v": 102,
}

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
GOLDEN = np.uint64(0x9E3779B97F4A7C15)
TID_MULT = np.uint64(0xD1B54A32D192ED03)
_CHUNK = 1 << 22


def _mix64(z):
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tid: int) -> np.uint64:
    s = _mix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
    with np.errstate(over="ignore"):
        t = np.uint64(tid) * TID_MULT
    return _mix64(np.array([s ^ t], dtype=np.uint64))[0]


def _stream(key: np.uint64, j: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return _mix64(key + (j.astype(np.uint64) + np.uint64(1)) * GOLDEN)


def uniform(seed: int, tid: int, shape, offset: int = 0) -> np.ndarray:
    """U[0, 1) float64 array of ``shape`` from stream (seed, tid), elements offset.. of the stream."""
    n = int(np.prod(shape))
    key = _key(seed, tid)
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        j = np.arange(offset + lo, offset + min(n, lo + _CHUNK), dtype=np.uint64)
        out[lo:lo + j.size] = (_stream(key, j) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return out.reshape(shape)


def normal(seed: int, tid: int, shape, scale: float = 1.0, offset: int = 0) -> np.ndarray:
    """N(0, scale^2) float64 array of ``shape`` from stream (seed, tid) via Box–Muller.

    Element i of the result is element ``offset + i`` of the tensor, so a
    slice of a large tensor can be produced without the rest.
    """
    n = int(np.prod(shape))
    key = _key(seed, tid)
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        i = np.arange(offset + lo, offset + min(n, lo + _CHUNK), dtype=np.uint64)
        h1 = _stream(key, i * np.uint64(2))
        h2 = _stream(key, i * np.uint64(2) + np.uint64(1))
        u1 = ((h1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (h2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        out[lo:lo + i.size] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (out * scale).reshape(shape)


def bf16_bits(x) -> np.ndarray:
    """uint16 bf16 bit patterns of ``x`` (float64 -> float32 -> bf16, both round-to-nearest-even)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact float64 values of uint16 bf16 bit patterns."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """float64 values of ``x`` after rounding to bf16."""
    return bf16_bits_to_f64(bf16_bits(x))


def uniform_row_normalised_mixing(seed: int, h: int, m: int) -> np.ndarray:
    """[h, m, m] mixing with U(0,1) entries, each row divided by its sum."""
    u = uniform(seed, TID["mix"], (h, m, m))
    return u / u.sum(axis=-1, keepdims=True)


def row_softmax_mixing(seed: int, h: int, m: int, diag_boost: float = 0.0) -> np.ndarray:
    """[h, m, m] mixing: each row is exp(l) / sum(exp(l)) of N(0,1) logits l plus ``diag_boost`` on the diagonal."""
    logits = normal(seed, TID["mix"], (h, m, m)) + diag_boost * np.eye(m)[None]
    e = np.exp(logits - logits.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)
