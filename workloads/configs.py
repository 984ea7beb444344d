"""The synthetic workloads: shapes, value distributions and seeds.

Each workload stands in for one workload shape of the source pages (the
datasets and trained weights behind them are not needed for a forward-path
kernel): DiT-S/2-like 64x64 latent token grids, a 256x256 high-resolution
token grid, long causal sequences with recurrent decode, and the 56x56
rank-augmented vision stage.  Seeds are ``SEED_BASE + index``.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .gen import (SEED_BASE, TID, bf16_bits, bf16_bits_to_f64, normal,
                  row_softmax_mixing, uniform_row_normalised_mixing)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # seed = SEED_BASE + index
    kind: str               # "mhla" | "causal" | "decode" | "rala"
    B: int
    H: int
    N: int
    d: int
    block: int = 0          # MHLA block size, or causal chunk
    dtype: str = "bf16"     # "f32" | "bf16"
    scale: float = 1.0      # std of Q, K, V
    mixing: str = "none"    # "uniform_rows" | "softmax_diag2" | "softmax" | "ones" | "none"
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def M(self) -> int:
        return self.N // self.block if self.block else 0

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * self.N


WORKLOADS = {
    # B1 H1 N256 d16, M = 4 blocks of 64, fp32, U(0,1) row-normalised mixing
    "tiny": Workload("tiny", 1, "mhla", 1, 1, 256, 16, 64, "f32", 1.0, "uniform_rows"),
    # DiT-S/2-like: 64x64 latent patch grid, row-major, M = 16 blocks of 256
    "dit": Workload("dit", 2, "mhla", 8, 6, 4096, 64, 256, "bf16", 0.125, "softmax_diag2"),
    # 256x256 token grid, M = 64 blocks of 1024, and the same inputs with M = 1
    "hires": Workload("hires", 3, "mhla", 1, 6, 65536, 64, 1024, "bf16", 0.125, "softmax"),
    "hires_m1": Workload("hires_m1", 3, "mhla", 1, 6, 65536, 64, 65536, "bf16", 0.125, "ones"),
    # long causal sequences, chunk 128
    "causal": Workload("causal", 4, "causal", 4, 16, 8192, 64, 128, "bf16", 0.125),
    # recurrent decode: batch 256 x 16 heads, 1024 steps after a 2048-token prefix
    "decode": Workload("decode", 4, "decode", 256, 16, 1024, 64, 0, "bf16", 0.125,
                       extra={"prefix": 2048}),
    # rank-augmented variant: 56x56 tokens, X [B, N, 64], W [64, 32]
    "rala": Workload("rala", 5, "rala", 64, 2, 3136, 32, 0, "bf16", 32 ** -0.5,
                     extra={"cx": 64}),
}


def _as_dtype(x64: np.ndarray, dtype: str):
    """(device representation, float64 values the oracle sees)."""
    if dtype == "bf16":
        bits = bf16_bits(x64)
        return bits, bf16_bits_to_f64(bits)
    f = np.asarray(x64, dtype=np.float32)
    return f, f.astype(np.float64)


def _heads_tensor(wl: Workload, tid: int, scale: float, heads, n: int, d: int, lead=None):
    """[B, H, n, d] tensor, or only the listed (b, h) slices stacked as [1, len(heads), n, d]."""
    if heads is None:
        return normal(wl.seed, tid, (wl.B, wl.H, n, d), scale)
    per = n * d
    out = np.empty((1, len(heads), n, d))
    for i, (b, h) in enumerate(heads):
        out[0, i] = normal(wl.seed, tid, (n, d), scale, offset=(b * wl.H + h) * per)
    return out


def make_mixing(wl: Workload) -> np.ndarray:
    """[H, M, M] float64 mixing matrix of a workload (rows: query blocks)."""
    if wl.mixing == "uniform_rows":
        return uniform_row_normalised_mixing(wl.seed, wl.H, wl.M)
    if wl.mixing == "softmax_diag2":
        return row_softmax_mixing(wl.seed, wl.H, wl.M, diag_boost=2.0)
    if wl.mixing == "softmax":
        return row_softmax_mixing(wl.seed, wl.H, wl.M)
    if wl.mixing == "ones":
        return np.ones((wl.H, wl.M, wl.M))
    raise ValueError(f"workload {wl.name} has no mixing")


def make_mhla_inputs(wl: Workload, heads=None) -> dict:
    """Q, K, V (and mixing for MHLA) of an MHLA or causal workload.

    Returns device representations (``q, k, v``: float32 or uint16 bf16 bits;
    ``mixing``: float32 [H, M, M]) and the float64 values the oracle consumes
    (``q64, k64, v64, mixing64``).  With ``heads`` = list of (b, h), only
    those slices are generated, as [1, len(heads), N, d] (mixing rows follow
    the listed heads).
    """
    out = {}
    for name in ("q", "k", "v"):
        x = _heads_tensor(wl, TID[name], wl.scale, heads, wl.N, wl.d)
        out[name], out[name + "64"] = _as_dtype(x, wl.dtype)
    if wl.kind == "mhla":
        mix = make_mixing(wl)
        if heads is not None:
            mix = mix[[h for _, h in heads]]
        out["mixing"] = mix.astype(np.float32)
        out["mixing64"] = out["mixing"].astype(np.float64)
    return out


def make_decode_inputs(wl: Workload, units=None, steps=None) -> dict:
    """Prefix K, V and per-step q, k, v of the decode workload.

    Shapes: ``prefix_k/v`` [P, U, d] and ``step_q/k/v`` [T, U, d] where the U
    = B*H (batch x head) units are flattened; ``units`` restricts to a list of
    unit indices.  Step t of unit u is element (t, u) of the step tensors.
    """
    u_all = wl.B * wl.H
    units = list(range(u_all)) if units is None else list(units)
    steps = wl.N if steps is None else steps
    p = wl.extra["prefix"]
    out = {}
    for name, tid, length in (("prefix_k", TID["prefix_k"], p), ("prefix_v", TID["prefix_v"], p),
                              ("step_q", TID["step_q"], steps), ("step_k", TID["step_k"], steps),
                              ("step_v", TID["step_v"], steps)):
        arr = np.empty((length, len(units), wl.d))
        for t in range(length):
            row = normal(wl.seed, tid, (u_all, wl.d), wl.scale, offset=t * u_all * wl.d)
            arr[t] = row[units]
        out[name], out[name + "64"] = _as_dtype(arr, wl.dtype)
    return out


def make_rala_inputs(wl: Workload, batches=None) -> dict:
    """Q, K, V [B, H, N, d], X [B, N, Cx], W [Cx, d] of the rank-augmented workload.

    Q, K, V ~ N(0, 1/d); X ~ N(0, 1); W ~ N(0, 1/Cx).  ``batches`` restricts
    to a list of batch indices.
    """
    cx = wl.extra["cx"]
    batches = list(range(wl.B)) if batches is None else list(batches)
    out = {}
    for name in ("q", "k", "v"):
        per = wl.H * wl.N * wl.d
        arr = np.stack([normal(wl.seed, TID[name], (wl.H, wl.N, wl.d), wl.scale, offset=b * per)
                        for b in batches])
        out[name], out[name + "64"] = _as_dtype(arr, wl.dtype)
    per_x = wl.N * cx
    x = np.stack([normal(wl.seed, TID["x"], (wl.N, cx), 1.0, offset=b * per_x) for b in batches])
    out["x"], out["x64"] = _as_dtype(x, wl.dtype)
    w = normal(wl.seed, TID["w"], (cx, wl.d), cx ** -0.5)
    out["w"], out["w64"] = _as_dtype(w, wl.dtype)
    return out
