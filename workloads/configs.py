"""The synthetic workloads: shapes, value distributions and seeds.

Each workload stands in for one workload shape of the source pages (the
datasets and trained weights behind them are not needed for a forward-path
kernel): DiT-S/2-like 64x64 latent token grids, a 256x256 high-resolution
token grid, long causal sequences with recurrent decode, and the 56x56
rank-augmented vision stage.  Seeds are ``SEED_BASE + index``.

``*_host`` functions return numpy arrays (device representation plus the
float64 values the oracle consumes) for the whole workload or a listed
subset; ``*_device`` functions return the full workload as torch tensors
generated on a device from the same streams.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .gen import (SEED_BASE, TID, bf16_bits, bf16_bits_to_f64, lower_row_normalised_mixing, normal, normal_at,
                  normal_device, row_softmax_mixing, uniform_row_normalised_mixing)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # seed = SEED_BASE + index
    kind: str               # "mhla" | "causal" | "decode" | "decode_steps" | "stream" | "rala" | "backward"
    B: int
    H: int
    N: int                  # tokens (decode: number of steps)
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
        if "M" in self.extra:
            return self.extra["M"]
        return self.N // self.block if self.block else 0

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * self.N


WORKLOADS = {
    # B1 H1 N256 d16, M = 4 blocks of 64, fp32, U(0,1) row-normalised mixing
    "tiny": Workload("tiny", 1, "mhla", 1, 1, 256, 16, 64, "f32", 1.0, "uniform_rows"),
    # DiT-S/2-like: 64x64 latent patch grid, row-major, M = 16 blocks of 256
    "dit": Workload("dit", 2, "mhla", 8, 6, 4096, 64, 256, "bf16", 0.125, "softmax_diag2"),
    # the same DiT-S/2-like inputs with 2-D blocks: the 64x64 grid cut into 4 x 4 tiles of 16x16
    "dit_grid": Workload("dit_grid", 2, "mhla", 8, 6, 4096, 64, 256, "bf16", 0.125, "softmax_diag2",
                         extra={"grid": (64, 64, 16, 16)}),
    # variants on the same inputs: no normaliser (MHLA §4.1), the ReLU feature map (notes §二)
    "dit_unnormalised": Workload("dit_unnormalised", 2, "mhla", 8, 6, 4096, 64, 256, "bf16", 0.125,
                                 "softmax_diag2", extra={"normalise": False}),
    "dit_relu": Workload("dit_relu", 2, "mhla", 8, 6, 4096, 64, 256, "bf16", 0.125, "softmax_diag2",
                         extra={"feature": "relu"}),
    # the backward of the DiT forward (dQ, dK, dV, dM) on the same inputs, dY ~ N(0, 1)
    "dit_backward": Workload("dit_backward", 2, "backward", 8, 6, 4096, 64, 256, "bf16", 0.125, "softmax_diag2"),
    # 256x256 token grid, M = 64 blocks of 1024, and the same inputs with M = 1
    "hires": Workload("hires", 3, "mhla", 1, 6, 65536, 64, 1024, "bf16", 0.125, "softmax"),
    "hires_m1": Workload("hires_m1", 3, "mhla", 1, 6, 65536, 64, 65536, "bf16", 0.125, "ones"),
    # long causal sequences, chunk 128
    "causal": Workload("causal", 4, "causal", 4, 16, 8192, 64, 128, "bf16", 0.125),
    # the causal inputs as causal MHLA: blocks of 128 (M = 64), a causal mixing matrix
    "causal_mhla": Workload("causal_mhla", 4, "causal", 4, 16, 8192, 64, 128, "bf16", 0.125,
                            "lower_uniform_rows"),
    # the causal inputs with RetNet decay gamma = 0.99 (notes §七)
    "causal_decay": Workload("causal_decay", 4, "causal", 4, 16, 8192, 64, 128, "bf16", 0.125,
                             extra={"gamma": 0.99}),
    # recurrent decode: batch 256 x 16 heads, 1024 steps after a 2048-token prefix
    "decode": Workload("decode", 4, "decode", 256, 16, 1024, 64, 0, "bf16", 0.125,
                       extra={"prefix": 2048}),
    # the same decode workload with all 1024 steps in one fused call (state held on chip)
    "decode_fused": Workload("decode_fused", 4, "decode_steps", 256, 16, 1024, 64, 0, "bf16", 0.125,
                             extra={"prefix": 2048}),
    # causal MHLA inference on the decode shape: 1024 tokens after a 2048-token prefix, blocks of
    # 128 (M = 24 for the 3072 tokens), a causal mixing matrix; N counts the streamed tokens
    "stream": Workload("stream", 4, "stream", 256, 16, 1024, 64, 128, "bf16", 0.125, "lower_uniform_rows",
                       extra={"prefix": 2048, "M": 24}),
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


def _torch_dtype(dtype: str):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def make_mixing(wl: Workload) -> np.ndarray:
    """[H, M, M] float64 mixing matrix of a workload (rows: query blocks), already float32-exact."""
    if wl.mixing == "uniform_rows":
        m = uniform_row_normalised_mixing(wl.seed, wl.H, wl.M)
    elif wl.mixing == "softmax_diag2":
        m = row_softmax_mixing(wl.seed, wl.H, wl.M, diag_boost=2.0)
    elif wl.mixing == "softmax":
        m = row_softmax_mixing(wl.seed, wl.H, wl.M)
    elif wl.mixing == "lower_uniform_rows":
        m = lower_row_normalised_mixing(wl.seed, wl.H, wl.M)
    elif wl.mixing == "ones":
        m = np.ones((wl.H, wl.M, wl.M))
    else:
        raise ValueError(f"workload {wl.name} has no mixing")
    return m.astype(np.float32).astype(np.float64)


# ------------------------------------------------------------ MHLA / causal
def mhla_host(wl: Workload, heads=None) -> dict:
    """Q, K, V (and mixing) of an MHLA or causal workload, on the host.

    ``q, k, v``: float32 arrays or uint16 bf16 bits; ``q64, k64, v64``: the
    float64 values the oracle consumes; ``mixing`` (float32 [H, M, M]) and
    ``mixing64`` for MHLA workloads.  With ``heads`` = list of (b, h) only
    those slices are produced, as [1, len(heads), N, d] (mixing rows follow
    the listed heads).
    """
    out = {}
    per = wl.N * wl.d
    for name in ("q", "k", "v") + (("dy",) if wl.kind == "backward" else ()):
        scale = 1.0 if name == "dy" else wl.scale
        if heads is None:
            x = normal(wl.seed, TID[name], (wl.B, wl.H, wl.N, wl.d), scale)
        else:
            x = np.stack([normal(wl.seed, TID[name], (wl.N, wl.d), scale, offset=(b * wl.H + h) * per)
                          for b, h in heads])[None]
        out[name], out[name + "64"] = _as_dtype(x, wl.dtype)
    if wl.mixing != "none":
        mix = make_mixing(wl)
        if heads is not None:
            mix = mix[[h for _, h in heads]]
        out["mixing64"] = mix
        out["mixing"] = mix.astype(np.float32)
    return out


def mhla_device(wl: Workload, device="cuda") -> dict:
    """The full MHLA / causal workload as device tensors (same values as :func:`mhla_host`)."""
    import torch
    dt = _torch_dtype(wl.dtype)
    names = ("q", "k", "v") + (("dy",) if wl.kind == "backward" else ())
    out = {name: normal_device(wl.seed, TID[name], (wl.B, wl.H, wl.N, wl.d), 1.0 if name == "dy" else wl.scale,
                               device=device, dtype=dt)
           for name in names}
    if wl.mixing != "none":
        out["mixing"] = torch.from_numpy(make_mixing(wl).astype(np.float32)).to(device)
    return out


# ------------------------------------------------------------------ decode
def _decode_index(u_all: int, d: int, steps, units) -> np.ndarray:
    t = np.asarray(steps, dtype=np.uint64)[:, None, None]
    u = np.asarray(units, dtype=np.uint64)[None, :, None]
    c = np.arange(d, dtype=np.uint64)[None, None, :]
    return (t * np.uint64(u_all * d) + u * np.uint64(d) + c)


def decode_host(wl: Workload, units, steps=None) -> dict:
    """Prefix K, V and per-step q, k, v of the decode workload for the listed units.

    The U = B*H (batch x head) units are flattened; a tensor of T rows is
    [T, U, d] with element (t, u, c) at flat index (t * U + u) * d + c.
    Returns [P or T, len(units), d] arrays (device representation and
    float64 values).
    """
    u_all = wl.B * wl.H
    steps = wl.N if steps is None else steps
    p = wl.extra["prefix"]
    out = {}
    for name, length in (("prefix_k", p), ("prefix_v", p), ("step_q", steps), ("step_k", steps),
                         ("step_v", steps)):
        idx = _decode_index(u_all, wl.d, range(length), units)
        x = normal_at(wl.seed, TID[name], idx.reshape(-1), wl.scale).reshape(idx.shape)
        out[name], out[name + "64"] = _as_dtype(x, wl.dtype)
    return out


def decode_device(wl: Workload, device="cuda", steps=None) -> dict:
    """Full decode workload on a device: prefix_k/v [P, B, H, d], step_q/k/v [T, B, H, d]."""
    steps = wl.N if steps is None else steps
    p = wl.extra["prefix"]
    dt = _torch_dtype(wl.dtype)
    out = {}
    for name, length in (("prefix_k", p), ("prefix_v", p), ("step_q", steps), ("step_k", steps),
                         ("step_v", steps)):
        out[name] = normal_device(wl.seed, TID[name], (length, wl.B, wl.H, wl.d), wl.scale,
                                  device=device, dtype=dt)
    return out


# -------------------------------------------------------------------- RALA
def rala_host(wl: Workload, batches=None) -> dict:
    """Q, K, V [B', H, N, d], X [B', N, Cx], W [Cx, d] of the rank-augmented workload.

    Q, K, V ~ N(0, 1/d); X ~ N(0, 1); W ~ N(0, 1/Cx).  ``batches`` restricts
    to a list of batch indices (B' = len(batches)).
    """
    cx = wl.extra["cx"]
    batches = list(range(wl.B)) if batches is None else list(batches)
    out = {}
    per = wl.H * wl.N * wl.d
    for name in ("q", "k", "v"):
        arr = np.stack([normal(wl.seed, TID[name], (wl.H, wl.N, wl.d), wl.scale, offset=b * per)
                        for b in batches])
        out[name], out[name + "64"] = _as_dtype(arr, wl.dtype)
    per_x = wl.N * cx
    x = np.stack([normal(wl.seed, TID["x"], (wl.N, cx), 1.0, offset=b * per_x) for b in batches])
    out["x"], out["x64"] = _as_dtype(x, wl.dtype)
    w = normal(wl.seed, TID["w"], (cx, wl.d), cx ** -0.5)
    out["w"], out["w64"] = _as_dtype(w, wl.dtype)
    return out


def rala_device(wl: Workload, device="cuda") -> dict:
    cx = wl.extra["cx"]
    dt = _torch_dtype(wl.dtype)
    out = {name: normal_device(wl.seed, TID[name], (wl.B, wl.H, wl.N, wl.d), wl.scale, device=device, dtype=dt)
           for name in ("q", "k", "v")}
    out["x"] = normal_device(wl.seed, TID["x"], (wl.B, wl.N, cx), 1.0, device=device, dtype=dt)
    out["w"] = normal_device(wl.seed, TID["w"], (cx, wl.d), cx ** -0.5, device=device, dtype=dt)
    return out
