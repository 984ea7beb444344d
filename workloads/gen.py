"""Counter-based random numbers and bf16 rounding for the synthetic workloads.

Generator: the SplitMix64 stream (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Output j of a stream with
seed ``key`` is ``mix64(key + (j + 1) * GOLDEN)``, so any element of any
tensor can be produced on its own.  Every tensor has its own stream:
``key = mix64(mix64(seed) ^ (tensor_id * TID_MULT))``.

* uniform[0,1): ``(h >> 11) * 2**-53`` of output j = flat index.
* standard normal (element i): Box–Muller, cosine branch, from outputs
  ``2i`` and ``2i + 1``: ``sqrt(-2 ln u1) cos(2 pi u2)`` with ``u1`` in (0, 1].

Two implementations of the same definition: numpy on the host (for the
slices the oracle checks) and torch on a device (for full-size tensors).

bf16 rounding: float64 -> float32 -> bf16, both round-to-nearest-even.
"""

from __future__ import annotations

import numpy as np

SEED_BASE = 20261202

# tensor ids inside one workload's stream family
TID = {
    "q": 1, "k": 2, "v": 3, "mix": 4, "x": 5, "w": 6,
    "prefix_k": 7, "prefix_v": 8,
    "step_q": 100, "step_k": 101, "step_v": 102,
    "dy": 9,
}

GOLDEN_INT = 0x9E3779B97F4A7C15
MIX1_INT = 0xBF58476D1CE4E5B9
MIX2_INT = 0x94D049BB133111EB
TID_MULT_INT = 0xD1B54A32D192ED03
_M64 = (1 << 64) - 1
_CHUNK = 1 << 22


# ------------------------------------------------------------ exact scalars
def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * MIX1_INT) & _M64
    z = ((z ^ (z >> 27)) * MIX2_INT) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int) -> int:
    """64-bit key of the stream of tensor ``tid`` under ``seed``."""
    return _mix64_int(_mix64_int(seed) ^ ((tid * TID_MULT_INT) & _M64))


# ------------------------------------------------------------------- numpy
def _mix64(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1_INT)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2_INT)
    return z ^ (z >> np.uint64(31))


def _stream(key: int, j: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + (j.astype(np.uint64) + np.uint64(1)) * np.uint64(GOLDEN_INT))


def uniform_at(seed: int, tid: int, idx) -> np.ndarray:
    """U[0,1) values of elements ``idx`` (flat indices) of tensor ``tid``."""
    idx = np.asarray(idx, dtype=np.uint64)
    return (_stream(stream_key(seed, tid), idx) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normal_at(seed: int, tid: int, idx, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values of elements ``idx`` (flat indices) of tensor ``tid``."""
    idx = np.asarray(idx, dtype=np.uint64)
    key = stream_key(seed, tid)
    h1 = _stream(key, idx * np.uint64(2))
    h2 = _stream(key, idx * np.uint64(2) + np.uint64(1))
    u1 = ((h1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * scale


def uniform(seed: int, tid: int, shape, offset: int = 0) -> np.ndarray:
    """U[0,1) float64 array of ``shape``: elements offset, offset+1, ... of tensor ``tid``."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = uniform_at(seed, tid, np.arange(offset + lo, offset + hi, dtype=np.uint64))
    return out.reshape(shape)


def normal(seed: int, tid: int, shape, scale: float = 1.0, offset: int = 0) -> np.ndarray:
    """N(0, scale^2) float64 array of ``shape``: elements offset, offset+1, ... of tensor ``tid``."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = normal_at(seed, tid, np.arange(offset + lo, offset + hi, dtype=np.uint64), scale)
    return out.reshape(shape)


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


def lower_row_normalised_mixing(seed: int, h: int, m: int) -> np.ndarray:
    """[h, m, m] causal mixing: U(0,1) + 0.05 entries at and below the diagonal, zero above,
    each row divided by its sum."""
    u = np.tril(uniform(seed, TID["mix"], (h, m, m)) + 0.05)
    return u / u.sum(axis=-1, keepdims=True)


# ------------------------------------------------------------------- torch
def _signed(x: int) -> int:
    x &= _M64
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(t, k: int):
    """Logical right shift of an int64 tensor holding uint64 bit patterns."""
    return (t >> k) & ((1 << (64 - k)) - 1)


def _mix64_t(z):
    z = (z ^ _lsr(z, 30)) * _signed(MIX1_INT)
    z = (z ^ _lsr(z, 27)) * _signed(MIX2_INT)
    return z ^ _lsr(z, 31)


def _stream_t(key: int, j):
    return _mix64_t((j + 1) * _signed(GOLDEN_INT) + _signed(key))


def normal_device(seed: int, tid: int, shape, scale: float = 1.0, offset: int = 0, device="cuda",
                  dtype=None):
    """Device version of :func:`normal` (same values): returns a float64 tensor, or ``dtype``.

    Converting the float64 result to bfloat16 goes through float32, matching
    :func:`bf16_bits` (both conversions round to nearest even).
    """
    import torch

    n = int(np.prod(shape))
    key = stream_key(seed, tid)
    out_dtype = torch.float64 if dtype is None else dtype
    out = torch.empty(n, dtype=out_dtype, device=device)
    chunk = 1 << 24
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        i = torch.arange(offset + lo, offset + hi, dtype=torch.int64, device=device)
        h1 = _stream_t(key, i * 2)
        h2 = _stream_t(key, i * 2 + 1)
        u1 = (_lsr(h1, 11).to(torch.float64) + 1.0) * 2.0 ** -53
        u2 = _lsr(h2, 11).to(torch.float64) * 2.0 ** -53
        x = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * np.pi * u2) * scale
        if out_dtype == torch.bfloat16:
            x = x.to(torch.float32)
        out[lo:hi] = x.to(out_dtype)
    return out.reshape(shape)
