"""A device-side wait that gives up: the failure path of the bounded waits.

The bf16 tensor-core forwards wait on other CTAs (per-head counters, grid
barriers) and on their own pipelines (mbarriers); every such wait has a time
limit, after which
the kernel lets its copies and MMAs in flight finish, raises the call's abort
flag, leaves the workspace counters at zero and latches MHLA_ERR_TIMEOUT in
the workspace.  ``mhla_debug_set_wait_limit_ns`` shortens the limit so that a
normal call runs into it; nothing faults or hangs: the waits just return.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_den, assert_close_y, to_f64
from test_parity_gpu import rand_inputs, rand_mixing
from token_level_head_gb300 import binding
from token_level_head_gb300.build import build_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_library()
    return binding.load()


@pytest.mark.parametrize("shape,path", [
    ((2, 3, 1152, 64, 128), "tcgen05_stream"),  # C = 9 chunks a head: per-head counters
    ((2, 2, 2048, 64, 256), "tcgen05"),         # C = 16: the three-pass kernel and its grid barriers
], ids=["stream", "three_pass"])
def test_wait_limit_gives_up_then_next_call_is_correct(shape, path):
    B, H, N, d, block = shape
    assert binding.mhla_forward_path(B, H, N, d, block, 0, torch.bfloat16) == path
    x = rand_inputs(700, (B, H, N, d), "bf16")
    mix_t, mix64 = rand_mixing(31, H, N // block)
    ws = binding.new_workspace(binding.mhla_workspace_bytes(B, H, N, d, block), "cuda")
    y = torch.zeros_like(x["q"])
    binding.mhla_debug_set_wait_limit_ns(1)  # any wait not already satisfied gives up
    try:
        binding.mhla_forward(x["q"], x["k"], x["v"], mix_t, y, block, workspace=ws)
        torch.cuda.synchronize()
    finally:
        binding.mhla_debug_set_wait_limit_ns(0)
    assert binding.mhla_query_status(ws) == binding.MHLA_ERR_TIMEOUT
    assert binding.mhla_query_status(ws) == binding.MHLA_OK  # reading the status clears it
    # the same workspace serves the next call: the counters were left at zero
    den = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    binding.mhla_forward(x["q"], x["k"], x["v"], mix_t, y, block, den_out=den, workspace=ws)
    assert binding.mhla_query_status(ws) == binding.MHLA_OK
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block)
    assert_close_y(to_f64(y), ref, "bf16")
    assert_close_den(to_f64(den), dref, "bf16")


def test_backward_wait_limit_gives_up_then_next_call_is_correct():
    """The tensor-core passes of the backward: with every wait at its shortest the call gives up,
    latches MHLA_ERR_TIMEOUT in its workspace, and the next call on the same workspace is right."""
    from test_backward_gpu import check, dm_term_magnitudes
    from test_parity_gpu import rounded
    from workloads import normal
    B, H, N, d, block = 2, 2, 512, 64, 128
    assert binding.mhla_backward_path(B, H, N, d, block, torch.bfloat16) == "tcgen05"
    x = rand_inputs(710, (B, H, N, d), "bf16")
    dy, dy64 = rounded(normal(711, 4, (B, H, N, d)), "bf16")
    mix_t, mix64 = rand_mixing(712, H, N // block)
    ws = binding.new_workspace(binding.mhla_backward_workspace_bytes(B, H, N, d, block), "cuda")
    grads = [torch.empty_like(x[n]) for n in "qkv"] + [torch.empty_like(mix_t)]
    binding.mhla_debug_set_wait_limit_ns(1)
    try:
        binding.mhla_backward(x["q"], x["k"], x["v"], mix_t, dy, *grads, block, workspace=ws)
        torch.cuda.synchronize()
    finally:
        binding.mhla_debug_set_wait_limit_ns(0)
    assert binding.mhla_query_status(ws) == binding.MHLA_ERR_TIMEOUT
    assert binding.mhla_query_status(ws) == binding.MHLA_OK
    binding.mhla_backward(x["q"], x["k"], x["v"], mix_t, dy, *grads, block, workspace=ws)
    assert binding.mhla_query_status(ws) == binding.MHLA_OK
    args = (x["q64"], x["k64"], x["v64"], mix64, block, dy64, 1e-6)
    check(tuple(to_f64(g) for g in grads), oracle.mhla_block_form_backward(*args), "bf16",
          dm_term_magnitudes(*args, absolute=True), "tcgen05")
