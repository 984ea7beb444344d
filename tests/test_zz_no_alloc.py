"""mhla_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (no allocator available to them, or no allocation allowed after
start-up) get the non-causal MHLA forward without a workspace; the library
keeps a fixed scratch array per GPU for it.  This file is collected last, so
a run that stops at its first failure has run every other test before it.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_DEN, TOL_Y, rel, slice_rel, to_f64
from token_level_head_gb300 import binding
from token_level_head_gb300.build import build_library
from workloads import WORKLOADS, mhla_device, normal, uniform

UNSUPPORTED = 2


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Validation happens on the host before any CUDA call; 64 heads x 65536 tokens need ~260 MB."""
    build_library()
    lib = binding.load()
    P = 1 << 20
    st = lib.mhla_forward_noalloc(P, 2 * P, 3 * P, 4 * P, 5 * (1 << 40), None, 8, 8, 65536, 64, 1024,
                                  1, 1e-6, None)
    assert st == UNSUPPORTED
    assert lib.mhla_forward_noalloc(P, 2 * P, 3 * P, 4 * P, 5 * P, None, 1, 1, 256, 48, 64, 1, 1e-6,
                                    None) == 1


def _inputs(seed, shape, dtype, block):
    B, H, N, d = shape
    t = {}
    for i, n in enumerate("qkv"):
        x = torch.from_numpy(normal(seed, i + 1, shape, d ** -0.5)).to("cuda")
        t[n] = x.to(torch.float32).to(dtype)
    u = uniform(seed, 4, (H, N // block, N // block)) + 0.05
    t["mixing"] = torch.from_numpy((u / u.sum(axis=-1, keepdims=True)).astype(np.float32)).to("cuda")
    return t


def _both(t, block):
    y_ref = torch.empty_like(t["q"])
    d_ref = torch.empty(t["q"].shape[:3], dtype=torch.float32, device="cuda")
    binding.mhla_forward(t["q"], t["k"], t["v"], t["mixing"], y_ref, block, den_out=d_ref)
    y = torch.empty_like(t["q"])
    den = torch.empty_like(d_ref)
    binding.mhla_forward_noalloc(t["q"], t["k"], t["v"], t["mixing"], y, block, den_out=den)
    torch.cuda.synchronize()
    return to_f64(y), to_f64(den), to_f64(y_ref), to_f64(d_ref)


@pytest.mark.gpu
def test_noalloc_matches_mhla_forward_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_library()
    wl = WORKLOADS["dit"]
    first = mhla_device(wl)
    second = _inputs(99, (wl.B, wl.H, wl.N, wl.d), torch.bfloat16, wl.block)
    for t in (first, second):   # two calls in a row on different data share the scratch
        y, den, y_ref, d_ref = _both(t, wl.block)
        assert np.all(np.isfinite(y))
        assert slice_rel(y, y_ref) <= TOL_Y["bf16"]
        assert rel(den, d_ref) <= TOL_DEN["bf16"]
    # fp32: mhla_forward runs the same kernels here, so the oracle checks it directly
    small = _inputs(7, (2, 3, 192, 16), torch.float32, 64)
    ref, dref = oracle.mhla_block_form(*(to_f64(small[n]) for n in ("q", "k", "v", "mixing")), 64)
    for _ in range(2):
        y, den, y_ref, d_ref = _both(small, 64)
        assert slice_rel(y, y_ref) <= TOL_Y["f32"]
        assert rel(den, d_ref) <= TOL_DEN["f32"]
        assert slice_rel(y, ref) <= TOL_Y["f32"]
        assert rel(den, dref) <= TOL_DEN["f32"]


@pytest.mark.gpu
def test_noalloc_small_call_after_large_call_sees_no_leftovers():
    """The scratch keeps the last call's contents; a smaller call after a larger one must not read them."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_library()
    big = _inputs(11, (4, 6, 2048, 64), torch.bfloat16, 128)
    _both(big, 128)
    small = _inputs(12, (1, 2, 512, 64), torch.bfloat16, 256)
    y, den, _, _ = _both(small, 256)
    ref, dref = oracle.mhla_block_form(*(to_f64(small[n]) for n in ("q", "k", "v", "mixing")), 256)
    assert slice_rel(y, ref) <= TOL_Y["bf16"]
    assert rel(den, dref) <= TOL_DEN["bf16"]
