"""The C-ABI library builds, loads, exports every declared symbol and rejects bad arguments.

Runs without a GPU: every call below fails host-side validation (or is an
empty no-op) before the library touches CUDA.
"""

import ctypes
import os
import re

import pytest
import torch

from token_level_head_gb300 import binding
from token_level_head_gb300.build import INCLUDE, build_library

OK, INVALID, UNSUPPORTED = 0, 1, 2
F32, BF16 = 0, 1


@pytest.fixture(scope="module")
def lib():
    build_library()
    return binding.load()


def declared_functions():
    text = open(os.path.join(INCLUDE, "mhla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)) - {"if"})


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "mhla_forward" in names and "linattn_decode_step" in names and "rala_forward" in names
    for name in names:
        assert hasattr(lib, name), name
        assert name in binding.EXPORTED, name


def test_status_strings(lib):
    for s in range(5):
        assert binding.status_string(s)
    assert binding.status_string(99) == "unknown status"


def test_workspace_queries(lib):
    assert binding.mhla_workspace_bytes(8, 6, 4096, 64, 256) > 0
    assert binding.mhla_workspace_bytes(8, 6, 4096, 48, 256) == 0       # d not supported
    assert binding.mhla_workspace_bytes(8, 6, 4096, 64, 300) == 0       # block does not divide N
    assert binding.mhla_workspace_bytes(8, 6, 4096, 64, 0) == 0
    small = binding.mhla_workspace_bytes(1, 1, 4096, 64, 256)
    big = binding.mhla_workspace_bytes(2, 1, 4096, 64, 256)
    assert 0 < small < big
    assert binding.rala_workspace_bytes(64, 2, 3136, 32, 64) > 0
    assert binding.rala_workspace_bytes(64, 2, 3136, 32, 60) == 0       # cx not a multiple of 16


P = 1 << 20  # fake, 256-byte-aligned "device" addresses; never dereferenced


def fwd(lib, q=P, k=2 * P, v=3 * P, mix=4 * P, y=5 * P, den=None, B=1, H=1, N=256, d=64,
        block=64, causal=0, dt=BF16, eps=1e-6, ws=8 * P, wsb=1 << 30):
    return lib.mhla_forward(q, k, v, mix, y, den, B, H, N, d, block, causal, dt, eps, ws, wsb, None)


def test_forward_argument_errors(lib):
    assert fwd(lib, d=48) == INVALID
    assert fwd(lib, block=100) == INVALID
    assert fwd(lib, block=0) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, dt=7) == INVALID
    assert fwd(lib, eps=-1.0) == INVALID
    assert fwd(lib, eps=float("nan")) == INVALID
    assert fwd(lib, eps=float("inf")) == INVALID
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, y=None) == INVALID
    assert fwd(lib, mix=None) == INVALID                    # non-causal MHLA needs the mixing
    assert fwd(lib, q=P + 8) == INVALID                     # misaligned
    assert fwd(lib, den=P * 40 + 4) == INVALID              # misaligned den_out
    assert fwd(lib, y=P + 4096) == INVALID                  # y overlaps q
    assert fwd(lib, y=P) == INVALID                         # y aliases q
    assert fwd(lib, ws=None) == INVALID
    assert fwd(lib, ws=8 * P + 16) == INVALID               # workspace not 256-aligned
    assert fwd(lib, wsb=16) == INVALID                      # workspace too small
    assert fwd(lib, causal=2) == INVALID


def test_empty_inputs_are_a_no_op(lib):
    assert fwd(lib, B=0) == OK
    assert fwd(lib, N=0, q=None, k=None, v=None, y=None) == OK
    assert lib.mhla_forward_causal(None, None, None, None, None, None, 0, 4, 128, 64, 64, BF16,
                                   1e-6, None, 0, None) == OK
    assert lib.linattn_decode_step(None, None, None, None, None, None, None, 0, 16, 64, BF16, 1e-6,
                                   None) == OK
    assert lib.rala_forward(None, None, None, None, None, None, 3, 2, 0, 32, 64, BF16, None, 0,
                            None) == OK


def test_decode_argument_errors(lib):
    def dec(q=P, k=2 * P, v=3 * P, S=4 * P, z=6 * P, out=7 * P, B=2, H=2, d=64, dt=BF16, eps=1e-6):
        return lib.linattn_decode_step(q, k, v, S, z, out, None, B, H, d, dt, eps, None)
    assert dec(d=24) == INVALID
    assert dec(S=None) == INVALID
    assert dec(z=4 * P + 64) == INVALID                    # z inside S
    assert dec(out=P) == INVALID                           # out aliases q
    assert dec(eps=-0.5) == INVALID
    assert dec(q=P + 2) == INVALID


def test_decode_steps_argument_errors(lib):
    def dec(q=P, k=2 * P, v=3 * P, S=4 * P, z=6 * P, out=7 * P, den=None, T=3, B=2, H=2, d=64, dt=BF16,
            eps=1e-6, gamma=1.0):
        return lib.linattn_decode_steps(q, k, v, S, z, out, den, T, B, H, d, dt, eps, gamma, None)
    assert dec(d=24) == INVALID
    assert dec(T=-1) == INVALID
    assert dec(S=None) == INVALID
    assert dec(z=4 * P + 64) == INVALID                    # z inside S
    assert dec(out=P) == INVALID                           # out aliases q
    assert dec(out=P + 2 * 2 * 64 * 2) == INVALID          # out overlaps step 1 of q
    assert dec(den=P) == INVALID                           # den_out aliases q
    assert dec(eps=-0.5) == INVALID
    assert dec(gamma=1.5) == INVALID
    assert dec(gamma=-0.1) == INVALID
    assert dec(gamma=float("nan")) == INVALID
    assert dec(q=P + 2) == INVALID
    assert dec(B=1 << 15, H=1 << 15) == UNSUPPORTED
    # empty: no steps, or no units
    assert dec(T=0, q=None, k=None, v=None, out=None) == OK
    assert dec(B=0, q=None, k=None, v=None, out=None, S=None, z=None) == OK


def test_grid_argument_errors_and_paths(lib):
    def grid(gh=64, gw=64, th=16, tw=16, d=64, dt=BF16, ws=8 * P, wsb=1 << 30, mix=4 * P, y=5 * P):
        return lib.mhla_forward_grid(P, 2 * P, 3 * P, mix, y, None, 2, 6, gh, gw, th, tw, d, dt, 1e-6,
                                     ws, wsb, None)
    assert grid(th=12) == INVALID                          # tiles do not cover the grid
    assert grid(tw=0) == INVALID
    assert grid(gw=0) == INVALID
    assert grid(d=40) == INVALID
    assert grid(mix=None) == INVALID
    assert grid(y=P) == INVALID                            # y aliases q
    assert grid(wsb=64) == INVALID                         # workspace too small
    assert grid(gh=0) == OK                                # no tokens
    path = lambda *a: binding.PATH_NAMES[lib.mhla_forward_grid_path(8, 6, *a)]  # noqa: E731
    assert path(64, 64, 16, 16, 64, BF16) == "tcgen05"
    assert path(16, 256, 1, 128, 64, BF16) == "tcgen05"    # 128-token rows of a tile
    assert path(8, 512, 2, 256, 64, BF16) == "tcgen05"
    assert path(64, 64, 16, 16, 64, F32) == "simt"
    assert path(64, 60, 16, 12, 64, BF16) == "simt"         # tile width neither divides nor is a multiple of 128
    assert path(64, 64, 4, 4, 64, BF16) == "simt"           # 16-token tiles
    assert path(64, 64, 12, 16, 64, BF16) == "none"


def test_locality_mixing_matches_the_oracle(lib):
    import numpy as np
    import oracle
    for bh, bw in [(1, 1), (1, 6), (4, 4), (3, 5), (8, 8)]:
        got = binding.locality_mixing(bh, bw).numpy()
        assert np.abs(got - oracle.locality_mixing_init(bh, bw)).max() < 1e-7
    assert lib.mhla_locality_mixing(None, 2, 2) == INVALID
    with pytest.raises(binding.MhlaError):
        binding.locality_mixing(0, 3)


def test_causal_stream_argument_errors(lib):
    def cs(q=P, S=4 * P, z=6 * P, out=7 * P, mix=8 * P, t0=0, T=5, B=2, H=2, d=64, block=64, M=4, eps=1e-6):
        return lib.mhla_causal_stream(q, 2 * P, 3 * P, mix, S, z, out, None, t0, T, B, H, d, block, M, BF16,
                                      eps, None)
    assert cs(d=48) == INVALID
    assert cs(t0=-1) == INVALID
    assert cs(t0=250, T=7) == INVALID                      # past the last block (4 x 64 tokens)
    assert cs(block=0) == INVALID
    assert cs(M=0) == INVALID
    assert cs(mix=None) == INVALID
    assert cs(out=P) == INVALID                            # out aliases q
    assert cs(z=4 * P + 64) == INVALID                     # z inside S
    assert cs(eps=float("inf")) == INVALID
    assert cs(T=0, q=None, out=None) == OK
    assert lib.mhla_causal_stream(None, None, None, None, None, None, None, None, 0, 4, 0, 2, 64, 64, 4, BF16,
                                  1e-6, None) == OK        # no units


def test_backward_argument_errors(lib):
    def bw(q=P, mix=4 * P, dy=5 * P, dq=6 * P, dk=7 * P, dv=8 * P, dm=9 * P, B=1, H=1, N=256, d=64, block=64,
           dt=BF16, eps=1e-6, ws=16 * P, wsb=1 << 30):
        return lib.mhla_backward(q, 2 * P, 3 * P, mix, dy, dq, dk, dv, dm, B, H, N, d, block, dt, eps, ws, wsb, None)
    assert binding.mhla_backward_workspace_bytes(1, 1, 256, 64, 64) > 0
    assert binding.mhla_backward_workspace_bytes(1, 1, 4096, 64, 32) == 0   # M = 128 blocks
    assert binding.mhla_backward_workspace_bytes(1, 1, 256, 48, 64) == 0    # d not supported
    assert bw(d=48) == INVALID
    assert bw(block=0) == INVALID
    assert bw(N=250) == INVALID                           # block does not divide N
    assert bw(N=4096, block=32) == UNSUPPORTED            # M = 128 > 64
    assert bw(mix=None) == INVALID
    assert bw(dq=P) == INVALID                            # dq aliases q
    assert bw(dk=6 * P) == INVALID                        # dk aliases dq
    assert bw(dm=4 * P + 16) == INVALID                   # dmixing inside the mixing
    assert bw(ws=None) == INVALID
    assert bw(ws=16 * P + 16) == INVALID                  # not 256-byte aligned
    assert bw(wsb=1024) == INVALID                        # too small
    assert bw(ws=6 * P) == INVALID                        # workspace over dq
    assert bw(eps=-1.0) == INVALID
    assert bw(dt=7) == INVALID
    assert bw(B=0, q=None, dq=None) == OK                 # nothing to do, no launch
    assert bw(N=0) == OK
    assert binding.mhla_backward_path(8, 6, 4096, 64, 256, torch.bfloat16) == "tcgen05"
    assert binding.mhla_backward_path(8, 6, 4096, 64, 256, torch.float32) == "simt"
    assert binding.mhla_backward_path(8, 6, 4096, 64, 64, torch.bfloat16) == "simt"   # blocks of half a chunk
    assert binding.mhla_backward_path(8, 6, 4096, 32, 256, torch.bfloat16) == "simt"
    assert binding.mhla_backward_path(1, 1, 4096, 64, 32, torch.bfloat16) == "none"   # M = 128


def test_options_argument_errors(lib):
    import ctypes
    def ex(feature=0, normalise=1, gamma=1.0, causal=0, mix=4 * P, B=2):
        opt = binding.MhlaOptions(feature, normalise, gamma)
        return lib.mhla_forward_ex(P, 2 * P, 3 * P, mix, 5 * P, None, B, 2, 256, 64, 64, causal, BF16, 1e-6,
                                   ctypes.byref(opt), 8 * P, 1 << 30, None)
    assert ex(feature=3) == INVALID
    assert ex(normalise=2) == INVALID
    assert ex(gamma=1.5) == INVALID
    assert ex(gamma=0.9) == INVALID                        # decay outside plain causal linear attention
    assert ex(gamma=0.9, causal=1) == INVALID              # causal MHLA (mixing given) has no decay
    assert ex(gamma=0.9, causal=1, mix=None, B=0) == OK    # plain causal, no units
    assert ex(feature=2, B=0) == OK
    path = lambda **kw: binding.mhla_forward_ex_path(8, 6, 4096, 64, 256, 0, 1, torch_bf16(), **kw)  # noqa: E731
    assert path() == "tcgen05" and path(normalise=False) == "tcgen05"
    assert path(feature="relu") == "simt" and path(feature="exp") == "simt"
    assert binding.mhla_forward_ex_path(4, 16, 8192, 64, 128, 1, 0, torch_bf16(), gamma=0.9) == "simt"
    assert binding.mhla_forward_ex_path(4, 16, 8192, 64, 128, 0, 1, torch_bf16(), gamma=0.9) == "none"
    with pytest.raises(ValueError, match="feature"):
        binding.mhla_forward_ex_path(1, 1, 256, 64, 64, 0, 1, torch_bf16(), feature="tanh")


def torch_bf16():
    import torch
    return torch.bfloat16


def test_rala_argument_errors(lib):
    def rala(cx=64, d=32, ws=8 * P, wsb=1 << 30, y=6 * P, x=4 * P):
        return lib.rala_forward(P, 2 * P, 3 * P, x, 5 * P, y, 2, 2, 3136, d, cx, BF16, ws, wsb, None)
    assert rala(cx=60) == INVALID
    assert rala(cx=512) == INVALID
    assert rala(d=20) == INVALID
    assert rala(wsb=8) == INVALID
    assert rala(y=P) == INVALID
    assert rala(cx=256, d=128) == UNSUPPORTED


def test_forward_path_query(lib):
    assert binding.PATH_NAMES[lib.mhla_forward_path(1, 1, 256, 16, 64, 0, F32)] == "simt"
    assert binding.PATH_NAMES[lib.mhla_forward_path(1, 1, 256, 48, 64, 0, F32)] == "none"
    assert binding.PATH_NAMES[lib.mhla_forward_path(4, 16, 8192, 64, 128, 1, BF16)] == "tcgen05"
    assert binding.PATH_NAMES[lib.mhla_forward_path(4, 16, 8192, 64, 100, 1, BF16)] == "none"
    assert binding.PATH_NAMES[lib.rala_forward_path(64, 2, 3136, 32, 64, BF16)] == "tcgen05"
    assert binding.PATH_NAMES[lib.rala_forward_path(64, 2, 3136, 32, 64, F32)] == "simt"
    assert binding.PATH_NAMES[lib.rala_forward_path(64, 3, 3136, 32, 64, BF16)] == "simt"
    assert binding.PATH_NAMES[lib.rala_forward_path(64, 2, 3100, 32, 64, BF16)] == "simt"
    assert binding.PATH_NAMES[lib.rala_forward_path(64, 2, 3136, 32, 60, BF16)] == "none"


def test_query_status_rejects_null(lib):
    assert lib.mhla_query_status(None, None) == INVALID


def test_launch_counter_starts_readable(lib):
    assert isinstance(binding.mhla_launch_count(), int)


def test_binding_rejects_mismatched_tensors():
    """Shape and dtype checks of the Python wrappers run before any device use (CPU tensors here)."""
    import torch
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16)
    ok_mix = torch.ones(2, 4, 4)
    cases = [
        dict(k=q[:, :1], msg="k: shape"),
        dict(v=q.float(), msg="v: dtype"),
        dict(y=torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16), msg="y: shape"),
        dict(mixing=torch.ones(2, 4, 4, dtype=torch.bfloat16), msg="mixing: dtype"),
        dict(mixing=torch.ones(2, 2, 2), msg="mixing: shape"),
        dict(den_out=torch.zeros(1, 2, 256, dtype=torch.float64), msg="den_out: dtype"),
    ]
    for c in cases:
        args = dict(k=q, v=q, y=q.clone(), mixing=ok_mix, den_out=None)
        msg = c.pop("msg")
        args.update(c)
        with pytest.raises(ValueError, match=msg):
            binding.mhla_forward(q, args["k"], args["v"], args["mixing"], args["y"], 64, den_out=args["den_out"])
    with pytest.raises(ValueError, match="CUDA"):  # consistent shapes, but not on a GPU
        binding.mhla_forward(q, q, q, ok_mix, q.clone(), 64)
    q3 = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="S: shape"):
        binding.linattn_decode_step(q3, q3, q3, torch.zeros(2, 64, 64), torch.zeros(1, 2, 64), q3.clone())
    q4 = torch.zeros(3, 1, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="den_out: shape"):
        binding.linattn_decode_steps(q4, q4, q4, torch.zeros(1, 2, 64, 64), torch.zeros(1, 2, 64), q4.clone(),
                                     den_out=torch.zeros(1, 2))
    with pytest.raises(ValueError, match="CUDA"):
        binding.linattn_decode_steps(q4, q4, q4, torch.zeros(1, 2, 64, 64), torch.zeros(1, 2, 64), q4.clone())
    with pytest.raises(ValueError, match="w: shape"):
        binding.rala_forward(q, q, q, torch.zeros(1, 256, 64, dtype=torch.bfloat16),
                             torch.zeros(64, 32, dtype=torch.bfloat16), q.clone())
