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
