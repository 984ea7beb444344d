"""GPU parity: the CUDA library through its C ABI against the float64 oracle.

Same seeded inputs on both sides (the oracle gets the dtype-rounded values).
Small shapes are compared element by element in full; the full-size
workloads run in the launch configuration the bench times and are compared
on sampled (batch, head) slices the oracle computes one by one, plus
properties checked over the whole output (finite, positive denominators).
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (TOL_Y, assert_close_den, assert_close_y, rel, slice_rel, to_device, to_f64,
                      torch_dtype)
from token_level_head_gb300 import binding
from token_level_head_gb300.build import build_library
from workloads import (WORKLOADS, bf16_bits, bf16_bits_to_f64, decode_device, decode_host,
                       mhla_device, mhla_host, normal, rala_device, rala_host, uniform)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_library()
    return binding.load()


def rounded(x64, dtype):
    """(device tensor, float64 values) of x64 rounded to dtype."""
    if dtype == "bf16":
        bits = bf16_bits(x64)
        return to_device(bits), bf16_bits_to_f64(bits)
    f = np.asarray(x64, np.float32)
    return to_device(f), f.astype(np.float64)


def rand_inputs(seed, shape, dtype, scale=None):
    d = shape[-1]
    scale = d ** -0.5 if scale is None else scale
    out = {}
    for i, name in enumerate("qkv"):
        out[name], out[name + "64"] = rounded(normal(seed, i + 1, shape, scale), dtype)
    return out


def rand_mixing(seed, h, m, lower=False):
    u = uniform(seed, 9, (h, m, m)) + 0.05
    if lower:
        u = np.tril(u)
    mix = (u / u.sum(axis=-1, keepdims=True)).astype(np.float32)
    return torch.from_numpy(mix).cuda(), mix.astype(np.float64)


def forward(q, k, v, mix, block, causal=0, eps=1e-6):
    y = torch.empty_like(q)
    den = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    binding.mhla_forward(q, k, v, mix, y, block, causal=causal, eps=eps, den_out=den)
    torch.cuda.synchronize()
    return to_f64(y), to_f64(den)


def forward_causal(q, k, v, mix, chunk, eps=1e-6):
    y = torch.empty_like(q)
    den = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    binding.mhla_forward_causal(q, k, v, mix, y, chunk, eps=eps, den_out=den)
    torch.cuda.synchronize()
    return to_f64(y), to_f64(den)


# ------------------------------------------------------------ non-causal MHLA
def test_tiny_workload_fp32():
    wl = WORKLOADS["tiny"]
    x = mhla_host(wl)
    q, k, v = (to_device(x[n]) for n in "qkv")
    mix = to_device(x["mixing"])
    y, den = forward(q, k, v, mix, wl.block)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)
    brute, dbrute = oracle.mhla_token_expansion(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)
    assert_close_y(y, ref, "f32")
    assert_close_y(y, brute, "f32")
    assert_close_den(den, dref, "f32")
    assert_close_den(den, dbrute, "f32")


SMALL = [  # B, H, N, d, block
    (2, 3, 192, 16, 64),
    (1, 2, 96, 32, 48),
    (1, 1, 128, 64, 1),
    (2, 2, 512, 64, 128),
    (1, 2, 256, 128, 256),
    (1, 3, 384, 64, 384),
    (3, 1, 1024, 64, 256),
    (1, 2, 768, 32, 256),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(shape, dtype):
    B, H, N, d, block = shape
    x = rand_inputs(100 + N + d, (B, H, N, d), dtype)
    mix_t, mix64 = rand_mixing(7 + block, H, N // block)
    y, den = forward(x["q"], x["k"], x["v"], mix_t, block)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block)
    assert_close_y(y, ref, dtype)
    assert_close_den(den, dref, dtype)


TC_SHAPES = [  # bf16, d = 64, blocks of whole 128-token tiles: the tcgen05 kernels
    # C = N / 128 a multiple of 16: the three-pass kernel
    (2, 3, 2048, 64, 128),    # M = 16, one chunk per block
    (1, 2, 4096, 64, 4096),   # M = 1 with 32 chunks (split block sums)
    (1, 1, 8192, 64, 128),    # M = 64, one chunk per block
    (2, 2, 6144, 64, 128),    # C = 48 partials (three K steps, two pairs a stage), M = 48
    (1, 3, 6144, 64, 256),    # M = 24: query blocks 24..31 of the mixing MMA are padding
    (1, 3, 4096, 64, 128),    # M = 32, C = 32
    (1, 2, 16384, 64, 2048),  # C = 128 > 64: the MIX MMAs in K chunks of 64 partials, M = 8
    (1, 1, 32768, 64, 32768), # M = 1 over C = 256 partials (z rows on CTAs of their own)
    # C not a multiple of 16: the stream kernel (partials zero-filled to 16)
    (1, 1, 128, 64, 128),     # one chunk, M = 1
    (3, 5, 640, 64, 128),     # odd head count, M = 5
    (2, 1, 1536, 64, 512),    # 4 chunks per block, C = 12
    (2, 3, 1152, 64, 384),    # 3 chunks per block, C = 9
    (4, 6, 1024, 64, 256),    # DiT-like blocks of 256 over 1024 tokens, 24 heads
    (1, 2, 8064, 64, 128),    # C = 63, M = 63: one tile per MIX item, 32 items a head
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tcgen05_shapes(shape):
    B, H, N, d, block = shape
    stream = (N // 128) % 16 != 0
    assert binding.mhla_forward_path(B, H, N, d, block, 0, torch.bfloat16) == ("tcgen05_stream" if stream else "tcgen05")
    x = rand_inputs(400 + N + B * H, (B, H, N, d), "bf16")
    mix_t, mix64 = rand_mixing(11 + block, H, N // block)
    y, den = forward(x["q"], x["k"], x["v"], mix_t, block)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block)
    assert_close_y(y, ref, "bf16")
    assert_close_den(den, dref, "bf16")


def test_bench_workloads_take_the_tensor_core_path():
    for name in ("dit", "hires", "hires_m1"):
        wl = WORKLOADS[name]
        assert binding.mhla_forward_path(wl.B, wl.H, wl.N, wl.d, wl.block, 0, torch.bfloat16) == "tcgen05"


def test_workspace_reuse_across_shapes_and_paths():
    """One zero-filled workspace, reused by SIMT and tcgen05 calls of different sizes, stays valid."""
    shapes = [(2, 2, 512, 64, 128, "bf16"), (1, 2, 256, 16, 64, "f32"), (4, 6, 1024, 64, 256, "bf16"),
              (1, 1, 256, 64, 128, "bf16"), (4, 6, 1024, 64, 256, "bf16")]
    big = max(binding.mhla_workspace_bytes(B, H, N, d, blk) for B, H, N, d, blk, _ in shapes)
    ws = binding.new_workspace(big, "cuda")
    for i, (B, H, N, d, blk, dt) in enumerate(shapes):
        x = rand_inputs(500 + i, (B, H, N, d), dt)
        mix_t, mix64 = rand_mixing(13 + i, H, N // blk)
        y = torch.empty_like(x["q"])
        den = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
        binding.mhla_forward(x["q"], x["k"], x["v"], mix_t, y, blk, den_out=den, workspace=ws)
        assert binding.mhla_query_status(ws) == 0
        ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, blk)
        assert_close_y(to_f64(y), ref, dt)
        assert_close_den(to_f64(den), dref, dt)


def test_extreme_values_fp32():
    """Large |Q|, |K| exercise both branches of phi far from 0 (exp underflow, big linear values)."""
    B, H, N, d, block = 1, 2, 256, 32, 64
    x = rand_inputs(31, (B, H, N, d), "f32", scale=6.0)
    mix_t, mix64 = rand_mixing(3, H, N // block)
    y, den = forward(x["q"], x["k"], x["v"], mix_t, block, eps=0.0)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block, eps=0.0)
    assert_close_y(y, ref, "f32")
    assert_close_den(den, dref, "f32")


# Edge cases on the bf16 tensor-core paths (both non-causal kernels): inputs far
# from zero (both branches of phi, exp of large negative values), eps = 0,
# identity mixing (per-block global linear attention, a closed form the
# oracle computes separately) and mixing with exact zeros.
TC_EDGE = [(2, 3, 2048, 64, 256), (2, 3, 1152, 64, 128)]  # three-pass kernel, stream kernel


@pytest.mark.parametrize("shape", TC_EDGE, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("scale", [4.0, 6.0])
def test_tcgen05_large_inputs_eps0(shape, scale):
    B, H, N, d, block = shape
    x = rand_inputs(600 + N, (B, H, N, d), "bf16", scale=scale)
    mix_t, mix64 = rand_mixing(17, H, N // block)
    y, den = forward(x["q"], x["k"], x["v"], mix_t, block, eps=0.0)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block, eps=0.0)
    assert_close_y(y, ref, "bf16")
    assert_close_den(den, dref, "bf16")


@pytest.mark.parametrize("shape", TC_EDGE, ids=lambda s: "x".join(map(str, s)))
def test_tcgen05_identity_mixing_is_blockwise_linear_attention(shape):
    B, H, N, d, block = shape
    M = N // block
    x = rand_inputs(610 + N, (B, H, N, d), "bf16")
    eye = np.broadcast_to(np.eye(M), (H, M, M)).astype(np.float32)
    y, den = forward(x["q"], x["k"], x["v"], torch.from_numpy(np.ascontiguousarray(eye)).cuda(), block)
    split = lambda a: a.reshape(B, H, M, block, d).transpose(0, 2, 1, 3, 4).reshape(B * M, H, block, d)  # noqa: E731
    ref, dref = oracle.global_linear_attention(split(x["q64"]), split(x["k64"]), split(x["v64"]))
    ref = ref.reshape(B, M, H, block, d).transpose(0, 2, 1, 3, 4).reshape(B, H, N, d)
    dref = dref.reshape(B, M, H, block).transpose(0, 2, 1, 3).reshape(B, H, N)
    assert_close_y(y, ref, "bf16")
    assert_close_den(den, dref, "bf16")


@pytest.mark.parametrize("shape", TC_EDGE, ids=lambda s: "x".join(map(str, s)))
def test_tcgen05_mixing_with_exact_zeros(shape):
    B, H, N, d, block = shape
    M = N // block
    x = rand_inputs(620 + N, (B, H, N, d), "bf16")
    u = uniform(21, 9, (H, M, M)) + 0.05
    u[uniform(21, 10, (H, M, M)) < 0.5] = 0.0
    u[np.arange(H)[:, None], np.arange(M)[None, :], np.arange(M)[None, :]] += 0.5  # no all-zero row
    mix = (u / u.sum(axis=-1, keepdims=True)).astype(np.float32)
    y, den = forward(x["q"], x["k"], x["v"], torch.from_numpy(mix).cuda(), block)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix.astype(np.float64), block)
    assert_close_y(y, ref, "bf16")
    assert_close_den(den, dref, "bf16")


@pytest.mark.parametrize("shape", [(2, 3, 2048, 64, 256), (2, 3, 1152, 64, 128)], ids=lambda s: "x".join(map(str, s)))
def test_tcgen05_without_den_out(shape):
    """The bench's call form: no den_out, a workspace reused by repeated calls."""
    B, H, N, d, block = shape
    x = rand_inputs(630 + N, (B, H, N, d), "bf16")
    mix_t, mix64 = rand_mixing(23, H, N // block)
    ws = binding.new_workspace(binding.mhla_workspace_bytes(B, H, N, d, block), "cuda")
    y = torch.empty_like(x["q"])
    for _ in range(3):
        binding.mhla_forward(x["q"], x["k"], x["v"], mix_t, y, block, workspace=ws)
    assert binding.mhla_query_status(ws) == 0
    ref, _ = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block)
    assert_close_y(to_f64(y), ref, "bf16")


def test_canary_regions_untouched():
    """Y, den_out and the workspace sit inside larger buffers filled with a pattern; nothing
    outside the regions the call owns may change (both tensor-core kernels and a SIMT shape)."""
    pad = 4096
    for shape in [(2, 3, 2048, 64, 256), (2, 3, 1152, 64, 128), (1, 2, 256, 32, 64)]:
        B, H, N, d, block = shape
        x = rand_inputs(640 + N, (B, H, N, d), "bf16")
        mix_t, mix64 = rand_mixing(29, H, N // block)
        n_y, n_d = B * H * N * d, B * H * N
        ybuf = torch.full((n_y + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
        dbuf = torch.full((n_d + 2 * pad,), -7.5, dtype=torch.float32, device="cuda")
        nws = binding.mhla_workspace_bytes(B, H, N, d, block)
        wbuf = torch.full((nws + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
        ws = wbuf[pad:pad + nws]
        ws.zero_()
        y = ybuf[pad:pad + n_y].view(torch.bfloat16).view(B, H, N, d)
        den = dbuf[pad:pad + n_d].view(B, H, N)
        binding.mhla_forward(x["q"], x["k"], x["v"], mix_t, y, block, den_out=den, workspace=ws)
        torch.cuda.synchronize()
        assert binding.mhla_query_status(ws) == 0
        for buf, fill in ((ybuf, 12345), (dbuf, -7.5), (wbuf, 0xA5)):
            assert bool((buf[:pad] == fill).all()) and bool((buf[-pad:] == fill).all()), f"canary {shape}"
        ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix64, block)
        assert_close_y(to_f64(y), ref, "bf16")
        assert_close_den(to_f64(den), dref, "bf16")


def test_device_generator_matches_host_generator():
    """The full-size tests generate Q, K, V on the device and the oracle's slices on the host:
    both must be the same bf16 values, bit for bit."""
    from workloads import normal_device
    shape = (2, 3, 1000, 64)
    for tid in (1, 2, 3):
        dev = normal_device(20261204, tid, shape, 0.125, device="cuda", dtype=torch.bfloat16)
        host = bf16_bits(normal(20261204, tid, shape, 0.125))
        assert np.array_equal(dev.view(torch.int16).cpu().numpy().view(np.uint16), host)
    devf = normal_device(20261205, 4, (7, 33), 1.0, device="cuda", dtype=torch.float32).cpu().numpy()
    assert np.array_equal(devf, normal(20261205, 4, (7, 33), 1.0).astype(np.float32))


@pytest.mark.parametrize("name", ["dit"])
def test_full_workload_all_heads(name):
    wl = WORKLOADS[name]
    dev = mhla_device(wl)
    y, den = forward(dev["q"], dev["k"], dev["v"], dev["mixing"], wl.block)
    x = mhla_host(wl)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)
    assert_close_y(y, ref, wl.dtype)
    assert_close_den(den, dref, wl.dtype)


def test_dit_grid_full_workload_all_heads():
    """The DiT-like workload with 2-D 16 x 16 blocks, in the bench's launch configuration, all
    48 heads against the oracle (blocks given token by token)."""
    wl = WORKLOADS["dit_grid"]
    gh, gw, th, tw = wl.extra["grid"]
    assert binding.mhla_forward_grid_path(wl.B, wl.H, gh, gw, th, tw, wl.d, torch.bfloat16) == "tcgen05"
    dev = mhla_device(wl)
    y = torch.empty_like(dev["q"])
    den = torch.empty(dev["q"].shape[:3], dtype=torch.float32, device="cuda")
    binding.mhla_forward_grid(dev["q"], dev["k"], dev["v"], dev["mixing"], y, (gh, gw), (th, tw), den_out=den)
    torch.cuda.synchronize()
    x = mhla_host(wl)
    ref, dref = oracle.mhla_block_form_ids(x["q64"], x["k64"], x["v64"], x["mixing64"],
                                           oracle.grid_block_ids(gh, gw, th, tw))
    assert_close_y(to_f64(y), ref, wl.dtype)
    assert_close_den(to_f64(den), dref, wl.dtype)


@pytest.mark.parametrize("name", ["hires", "hires_m1"])
def test_full_workload_every_head(name):
    wl = WORKLOADS[name]
    dev = mhla_device(wl)
    y, den = forward(dev["q"], dev["k"], dev["v"], dev["mixing"], wl.block)
    assert np.all(np.isfinite(y)) and np.all(den > 0)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    x = mhla_host(wl, heads=heads)
    ref, dref = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)
    for i, (b, h) in enumerate(heads):
        assert_close_y(y[b, h][None, None], ref[0, i][None, None], wl.dtype, what=f"Y[{b},{h}]")
        assert_close_den(den[b, h], dref[0, i], wl.dtype, what=f"den[{b},{h}]")


def test_m1_equals_all_ones_mixing():
    """Global linear attention two ways on the GPU path: M = 1, and all-ones mixing over M = 8 blocks."""
    x = rand_inputs(55, (1, 2, 1024, 64), "bf16")
    y1, d1 = forward(x["q"], x["k"], x["v"], torch.ones(2, 1, 1, device="cuda"), 1024)
    y8, d8 = forward(x["q"], x["k"], x["v"], torch.ones(2, 8, 8, device="cuda"), 128)
    ref, dref = oracle.global_linear_attention(x["q64"], x["k64"], x["v64"])
    for y, den in ((y1, d1), (y8, d8)):
        assert_close_y(y, ref, "bf16")
        assert_close_den(den, dref, "bf16")


def test_deterministic():
    wl = WORKLOADS["dit"]
    dev = mhla_device(wl)
    outs = []
    for _ in range(2):
        y = torch.empty_like(dev["q"])
        binding.mhla_forward(dev["q"], dev["k"], dev["v"], dev["mixing"], y, wl.block)
        torch.cuda.synchronize()
        outs.append(y.view(torch.int16).clone())
    assert torch.equal(outs[0], outs[1])


def test_empty_batch_is_a_no_op():
    q = torch.empty(0, 2, 256, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(q)
    ws = binding.new_workspace(256, "cuda")
    binding.mhla_forward(q, q, q, torch.ones(2, 4, 4, device="cuda"), y, 64, workspace=ws)
    assert binding.mhla_query_status(ws) == 0


# --------------------------------------------------------------------- causal
CAUSAL = [  # B, H, N, d, chunk
    (2, 2, 256, 16, 64),
    (1, 2, 384, 64, 128),
    (1, 1, 256, 32, 16),
    (1, 2, 512, 64, 512),
    (2, 1, 256, 128, 128),
    (1, 1, 64, 64, 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", CAUSAL, ids=lambda s: "x".join(map(str, s)))
def test_causal_small(shape, dtype):
    B, H, N, d, chunk = shape
    x = rand_inputs(200 + N + d, (B, H, N, d), dtype)
    y, den = forward_causal(x["q"], x["k"], x["v"], None, chunk)
    ref, dref = oracle.causal_chunked(x["q64"], x["k64"], x["v64"], chunk)
    assert_close_y(y, ref, dtype)
    assert_close_den(den, dref, dtype)
    if N <= 256:
        brute, dbrute = oracle.causal_bruteforce(x["q64"], x["k64"], x["v64"])
        assert_close_y(y, brute, dtype)
        assert_close_den(den, dbrute, dtype)


# bf16, d = 64, N a multiple of 128: the tensor-core causal kernels.  The
# chunks of all heads are cut into one contiguous segment per CTA, so these
# shapes put head starts at every position inside a segment and spread heads
# over several CTAs.
CAUSAL_TC = [  # B, H, N, chunk
    (4, 100, 128, 128),   # one chunk per head: several whole heads per CTA
    (3, 100, 256, 64),    # two chunks per head
    (1, 5, 10240, 128),   # 80 chunks per head, each head over ~30 CTAs
    (1, 1, 128, 128),     # a single chunk
]


@pytest.mark.parametrize("shape", CAUSAL_TC, ids=lambda s: "x".join(map(str, s)))
def test_causal_tcgen05_shapes(shape):
    B, H, N, chunk = shape
    assert binding.mhla_forward_path(B, H, N, 64, chunk, 1, torch.bfloat16) == "tcgen05"
    x = rand_inputs(300 + N + H, (B, H, N, 64), "bf16")
    y, den = forward_causal(x["q"], x["k"], x["v"], None, chunk)
    ref, dref = oracle.causal_chunked(x["q64"], x["k64"], x["v64"], 128)
    assert_close_y(y, ref, "bf16")
    assert_close_den(den, dref, "bf16")


def test_causal_tcgen05_repeat_is_deterministic():
    x = rand_inputs(41, (2, 3, 1024, 64), "bf16")
    y1, d1 = forward_causal(x["q"], x["k"], x["v"], None, 128)
    y2, d2 = forward_causal(x["q"], x["k"], x["v"], None, 128)
    assert np.array_equal(y1, y2) and np.array_equal(d1, d2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_causal_mhla_with_mixing(dtype):
    B, H, N, d, chunk = 1, 2, 256, 32, 64
    x = rand_inputs(77, (B, H, N, d), dtype)
    mix_t, mix64 = rand_mixing(5, H, N // chunk, lower=True)
    y, den = forward_causal(x["q"], x["k"], x["v"], mix_t, chunk)
    ref, dref = oracle.causal_mhla_bruteforce(x["q64"], x["k64"], x["v64"], mix64, chunk)
    assert_close_y(y, ref, dtype)
    assert_close_den(den, dref, dtype)
    # mhla_forward(causal=1) is the same computation
    y2, den2 = forward(x["q"], x["k"], x["v"], mix_t, chunk, causal=1)
    assert np.array_equal(y2, y) and np.array_equal(den2, den)


CAUSAL_MHLA_TC = [  # B, H, N (d = 64, chunk = block = 128, bf16)
    (1, 2, 1024),   # M = 8
    (2, 3, 2048),   # M = 16
    (2, 2, 4096),   # M = 32
    (1, 4, 8192),   # M = 64
    (3, 1, 384),    # M = 3
]


@pytest.mark.parametrize("shape", CAUSAL_MHLA_TC, ids=lambda s: "x".join(map(str, s)))
def test_causal_mhla_tcgen05(shape):
    """Causal MHLA with a lower-triangular mixing on the tensor cores (the MHLA kernel's prefix
    pass, then the causal output kernel) against the oracle's chunk form; entries above the
    diagonal are large and must not reach the result."""
    B, H, N = shape
    d, chunk = 64, 128
    assert binding.mhla_forward_ex_path(B, H, N, d, chunk, 1, 1, torch.bfloat16) == "tcgen05"
    x = rand_inputs(780 + N, (B, H, N, d), "bf16")
    M = N // chunk
    u = np.tril(uniform(781, 9, (H, M, M)) + 0.05)
    mix = u / u.sum(axis=-1, keepdims=True) + np.triu(np.full((M, M), 5.0), 1)
    mix_t = torch.from_numpy(mix.astype(np.float32)).cuda()
    y, den = forward_causal(x["q"], x["k"], x["v"], mix_t, chunk)
    ref, dref = oracle.causal_mhla_chunked(x["q64"], x["k64"], x["v64"], np.tril(mix.astype(np.float32)), chunk)
    assert_close_y(y, ref, "bf16")
    assert_close_den(den, dref, "bf16")


def test_causal_mhla_tcgen05_full_size_sampled_heads():
    """The causal workload's shape (B4 H16 N8192, M = 64) with a causal mixing, 8 heads against
    the oracle; every output finite."""
    wl = WORKLOADS["causal"]
    dev = mhla_device(wl)
    M = wl.N // wl.block
    u = np.tril(uniform(790, 9, (wl.H, M, M)) + 0.05)
    mix = (u / u.sum(axis=-1, keepdims=True)).astype(np.float32)
    y, den = forward_causal(dev["q"], dev["k"], dev["v"], torch.from_numpy(mix).cuda(), wl.block)
    assert np.all(np.isfinite(y)) and np.all(den > 0)
    heads = [(0, 0), (0, 15), (1, 3), (1, 8), (2, 11), (2, 6), (3, 1), (3, 15)]
    x = mhla_host(wl, heads=heads)
    mixh = mix[[h for _, h in heads]].astype(np.float64)
    ref, dref = oracle.causal_mhla_chunked(x["q64"], x["k64"], x["v64"], mixh, wl.block)
    for i, (b, h) in enumerate(heads):
        assert_close_y(y[b, h][None, None], ref[0, i][None, None], wl.dtype, what=f"Y[{b},{h}]")
        assert_close_den(den[b, h], dref[0, i], wl.dtype, what=f"den[{b},{h}]")


def test_causal_full_workload_every_head():
    wl = WORKLOADS["causal"]
    dev = mhla_device(wl)
    y, den = forward_causal(dev["q"], dev["k"], dev["v"], None, wl.block)
    assert np.all(np.isfinite(y)) and np.all(den > 0)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    x = mhla_host(wl, heads=heads)
    ref, dref = oracle.causal_chunked(x["q64"], x["k64"], x["v64"], wl.block)
    for i, (b, h) in enumerate(heads):
        assert_close_y(y[b, h][None, None], ref[0, i][None, None], wl.dtype, what=f"Y[{b},{h}]")
        assert_close_den(den[b, h], dref[0, i], wl.dtype, what=f"den[{b},{h}]")


# --------------------------------------------------------------------- decode
def decode_run(S, z, qs, ks, vs, eps=1e-6):
    """Runs T steps on the GPU; returns per-step outputs and denominators (float64)."""
    outs, dens = [], []
    for t in range(qs.shape[0]):
        out = torch.empty_like(qs[t])
        den = torch.empty(qs.shape[1:-1], dtype=torch.float32, device=qs.device)
        binding.linattn_decode_step(qs[t], ks[t], vs[t], S, z, out, eps=eps, den_out=den)
        outs.append(out)
        dens.append(den)
    torch.cuda.synchronize()
    return to_f64(torch.stack(outs)), to_f64(torch.stack(dens))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_decode_small(d, dtype):
    B, H, T, P = 3, 5, 12, 40
    pk = normal(9, 1, (P, B, H, d), d ** -0.5)
    pv = normal(9, 2, (P, B, H, d), d ** -0.5)
    kf = oracle.phi(pk)
    s0 = np.einsum("pbhc,pbhe->bhce", kf, pv).astype(np.float32)
    z0 = kf.sum(axis=0).astype(np.float32)
    steps = {n: rounded(normal(9, 3 + i, (T, B, H, d), d ** -0.5), dtype) for i, n in enumerate("qkv")}
    S, z = torch.from_numpy(s0).cuda(), torch.from_numpy(z0).cuda()
    outs, dens = decode_run(S, z, steps["q"][0], steps["k"][0], steps["v"][0])
    ref, dref, s_t, z_t = oracle.decode_steps(s0, z0, steps["q"][1], steps["k"][1], steps["v"][1])
    assert_close_y(outs.reshape(T * B, H, d)[:, :, None], ref.reshape(T * B, H, d)[:, :, None], dtype)
    assert_close_den(dens, dref, dtype)
    assert_close_y(to_f64(S), s_t, "f32", what="state S")
    assert rel(to_f64(z), z_t) < 1e-5


def test_decode_full_workload_sampled_units():
    wl = WORKLOADS["decode"]
    B, H, d = wl.B, wl.H, wl.d
    dev = decode_device(wl)
    # initial state: the prefix summary.  Computed on the device by torch for
    # every unit, then overwritten by the oracle's value for the checked units.
    kf = torch.where(dev["prefix_k"].float() > 0, dev["prefix_k"].float() + 1, torch.exp(dev["prefix_k"].float()))
    S = torch.einsum("pbhc,pbhe->bhce", kf, dev["prefix_v"].float()).contiguous()
    z = kf.sum(dim=0).contiguous()
    units = list(range(0, B * H, 64)) + [B * H - 1]  # every 64th unit and the last: 65 units
    host = decode_host(wl, units)
    s0 = np.einsum("puc,pue->uce", oracle.phi(host["prefix_k64"]), host["prefix_v64"]).astype(np.float32)
    z0 = oracle.phi(host["prefix_k64"]).sum(axis=0).astype(np.float32)
    Sf, zf = S.view(B * H, d, d), z.view(B * H, d)
    for i, u in enumerate(units):
        Sf[u] = torch.from_numpy(s0[i]).cuda()
        zf[u] = torch.from_numpy(z0[i]).cuda()
    T = wl.N
    outs = torch.empty(T, len(units), d, dtype=torch.float32, device="cuda")
    dens = torch.empty(T, len(units), dtype=torch.float32, device="cuda")
    sel = torch.tensor(units, device="cuda")
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    den = torch.empty(B, H, dtype=torch.float32, device="cuda")
    for t in range(T):
        binding.linattn_decode_step(dev["step_q"][t], dev["step_k"][t], dev["step_v"][t], S, z, out,
                                    den_out=den)
        outs[t] = out.view(B * H, d)[sel].float()
        dens[t] = den.view(B * H)[sel]
    torch.cuda.synchronize()
    ref, dref, s_t, _ = oracle.decode_steps(s0, z0, host["step_q64"], host["step_k64"], host["step_v64"])
    assert_close_y(to_f64(outs).transpose(1, 0, 2)[:, None], ref.transpose(1, 0, 2)[:, None], "bf16")
    assert_close_den(to_f64(dens), dref, "bf16")
    assert_close_y(to_f64(Sf[sel])[:, None], s_t[:, None], "f32", what="state S")


# ------------------------------------------------ phi on the tensor-core paths
def bf16_grid_values(lo=-20.0, hi=20.0, tiny=1e-3):
    """Every bf16 value x with tiny <= |x| <= 20 in [lo, hi], and 0 (about 3.9 thousand), as float64."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite patterns only
    x = bf16_bits_to_f64(bits)
    keep = (x >= lo) & (x <= hi) & ((np.abs(x) >= tiny) | (x == 0))
    return np.unique(x[keep])


def phi_bound(x):
    """|phi_gpu - phi| / phi the kernels must meet: the base-2 exponential (2^-21 relative, with
    margin) plus the rounding of x log2 e (|x| 2^-24 relative in the exponent) and of the fp32
    sums around it (2^-23)."""
    return 2.0 ** -21 + np.abs(x) * 2.0 ** -23


@pytest.mark.parametrize("path", ["tcgen05", "tcgen05_stream", "causal_tcgen05"])
def test_phi_on_the_tensor_core_paths(path):
    """phi(x) for every bf16 x with 1e-3 <= |x| <= 20 (and 0), read back through the fp32
    denominator: Q = 0 (phi = 1), identity mixing, eps = 0, and in each block one key element x
    with every other key element -100 (phi flushes to 0), so den = phi(x) up to the bound above."""
    xs = bf16_grid_values()
    if path == "causal_tcgen05":
        N, block, per = 128, 128, 1          # one value per head, at its first token
    elif path == "tcgen05":
        N, block, per = 2048, 128, 16        # C = 16: the three-pass kernel
    else:
        N, block, per = 1152, 128, 9         # C = 9: the stream kernel
    heads = -(-len(xs) // per)
    vals = np.resize(xs, heads * per)        # pad by repeating
    d = 64
    k = np.full((1, heads, N, d), -100.0)
    for j in range(per):
        k[0, :, j * block, 0] = vals[j::per]
    kt = to_device(bf16_bits(k))
    q = torch.zeros(1, heads, N, d, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(q)
    y = torch.empty_like(q)
    den = torch.empty(1, heads, N, dtype=torch.float32, device="cuda")
    eps = 0.0
    if path == "causal_tcgen05":
        assert binding.mhla_forward_path(1, heads, N, d, block, 1, torch.bfloat16) == "tcgen05"
        binding.mhla_forward_causal(q, kt, v, None, y, block, eps=eps, den_out=den)
        got = to_f64(den)[0, :, 0]
    else:
        assert binding.mhla_forward_path(1, heads, N, d, block, 0, torch.bfloat16) == path
        mix = torch.eye(N // block, dtype=torch.float32, device="cuda").expand(heads, -1, -1).contiguous()
        binding.mhla_forward(q, kt, v, mix, y, block, eps=eps, den_out=den)
        got = to_f64(den)[0][:, ::block].reshape(-1)
    torch.cuda.synchronize()
    ref = oracle.phi(vals)
    err = np.abs(got - ref) / ref
    if path == "causal_tcgen05":
        # the causal denominator sums fp32 phi(K) (an in-chunk prefix beside the MMAs)
        bound = phi_bound(vals)
    else:
        # z comes out of the summary MMA, whose B operand is phi(K) rounded to bf16: den is
        # that rounding of the fp32 phi, so |error| <= half a bf16 ulp (2^-8 relative) + the above,
        # and it equals the bf16 rounding of the exact phi except within 2^-21 of a tie
        bound = 2.0 ** -8 + phi_bound(vals)
        exact = bf16_bits_to_f64(bf16_bits(ref))
        assert np.mean(got == exact) > 0.999, f"{np.mean(got == exact):.4f} equal to the rounded phi"
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), f"x = {vals[worst]}: relative error {err[worst]:.3e}"


# ------------------------------------------ variants: phi, normaliser, decay
VARIANT_SHAPES = [  # B, H, N, d, block, dtype
    (2, 3, 192, 16, 64, "f32"),
    (1, 2, 512, 64, 128, "bf16"),
    (2, 2, 256, 32, 256, "f32"),
]


@pytest.mark.parametrize("feature", ["relu", "exp"])
@pytest.mark.parametrize("normalise", [True, False])
@pytest.mark.parametrize("shape", VARIANT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_feature_variants_noncausal(shape, feature, normalise):
    B, H, N, d, block, dtype = shape
    assert binding.mhla_forward_ex_path(B, H, N, d, block, 0, 1, torch_dtype(dtype), feature=feature) == "simt"
    x = rand_inputs(700 + N + d, (B, H, N, d), dtype)
    mix_t, mix64 = rand_mixing(701, H, N // block)
    y = torch.empty_like(x["q"])
    den = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    binding.mhla_forward_ex(x["q"], x["k"], x["v"], mix_t, y, block, feature=feature, normalise=normalise,
                            den_out=den)
    torch.cuda.synchronize()
    ref, dref = oracle.mhla_block_form_feature(x["q64"], x["k64"], x["v64"], mix64, block, feature, 1e-6,
                                               normalise)
    assert_close_y(to_f64(y), ref, dtype)
    assert_close_den(to_f64(den), dref, dtype)


# normaliser-free output on every kernel family: SIMT, tcgen05, tcgen05 stream, causal tcgen05
UNNORM = [  # B, H, N, d, block, causal, dtype, path
    (2, 3, 256, 32, 64, 0, "f32", "simt"),
    (2, 6, 4096, 64, 256, 0, "bf16", "tcgen05"),
    (2, 3, 1152, 64, 384, 0, "bf16", "tcgen05_stream"),
    (2, 4, 2048, 64, 128, 1, "bf16", "tcgen05"),
    (1, 2, 384, 32, 64, 1, "f32", "simt"),
]


@pytest.mark.parametrize("shape", UNNORM, ids=lambda s: "x".join(map(str, s[:6])) + f"-{s[6]}")
def test_normaliser_free_output(shape):
    B, H, N, d, block, causal, dtype, path = shape
    assert binding.mhla_forward_ex_path(B, H, N, d, block, causal, 0 if causal else 1, torch_dtype(dtype),
                                        normalise=False) == path
    x = rand_inputs(720 + N + d, (B, H, N, d), dtype)
    mix_t, mix64 = (None, None) if causal else rand_mixing(721, H, N // block)
    y = torch.empty_like(x["q"])
    den = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    binding.mhla_forward_ex(x["q"], x["k"], x["v"], mix_t, y, block, causal=causal, normalise=False, den_out=den)
    torch.cuda.synchronize()
    if causal:
        ref, dref = oracle.causal_variant_bruteforce(x["q64"], x["k64"], x["v64"], "elu1", 1.0, 1e-6, False)
    else:
        ref, dref = oracle.mhla_block_form_feature(x["q64"], x["k64"], x["v64"], mix64, block, "elu1", 1e-6,
                                                   False)
    assert_close_y(to_f64(y), ref, dtype)
    assert_close_den(to_f64(den), dref, dtype)


@pytest.mark.parametrize("gamma", [0.9, 0.99, 0.0])
@pytest.mark.parametrize("shape", [(2, 2, 320, 32, 64, "f32"), (1, 3, 512, 64, 128, "bf16"),
                                   (1, 2, 300, 16, 60, "f32")], ids=lambda s: "x".join(map(str, s)))
def test_causal_decay(shape, gamma):
    """Plain causal linear attention with RetNet decay, chunked on the SIMT kernels, against the
    explicit decayed weights; the result must not depend on the chunk."""
    B, H, N, d, chunk, dtype = shape
    assert binding.mhla_forward_ex_path(B, H, N, d, chunk, 1, 0, torch_dtype(dtype), gamma=gamma) == "simt"
    x = rand_inputs(740 + N + d, (B, H, N, d), dtype)
    y = torch.empty_like(x["q"])
    den = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    binding.mhla_forward_ex(x["q"], x["k"], x["v"], None, y, chunk, causal=1, gamma=gamma, den_out=den)
    torch.cuda.synchronize()
    ref, dref = oracle.causal_variant_bruteforce(x["q64"], x["k64"], x["v64"], "elu1", gamma)
    assert_close_y(to_f64(y), ref, dtype)
    assert_close_den(to_f64(den), dref, dtype)


def test_causal_decay_with_relu_and_no_normaliser():
    B, H, N, d, chunk = 1, 2, 256, 32, 64
    x = rand_inputs(760, (B, H, N, d), "f32")
    y = torch.empty_like(x["q"])
    binding.mhla_forward_ex(x["q"], x["k"], x["v"], None, y, chunk, causal=1, gamma=0.95, feature="relu",
                            normalise=False)
    torch.cuda.synchronize()
    ref, _ = oracle.causal_variant_recurrent(x["q64"], x["k64"], x["v64"], "relu", 0.95, 1e-6, False)
    assert_close_y(to_f64(y), ref, "f32")


# ----------------------------------------------------------- 2-D grid blocks
GRID = [  # B, H, grid_h, grid_w, tile_h, tile_w, d, dtype, mixing, path
    (2, 3, 12, 20, 3, 5, 16, "f32", "random", "simt"),
    (1, 2, 16, 16, 4, 8, 32, "bf16", "locality", "simt"),
    (1, 1, 8, 24, 8, 3, 64, "bf16", "random", "simt"),
    (2, 3, 64, 64, 16, 16, 64, "bf16", "locality", "tcgen05"),     # the DiT latent grid, 4 x 4 tiles
    (1, 2, 32, 64, 8, 16, 64, "bf16", "random", "tcgen05"),
    (1, 2, 16, 256, 1, 128, 64, "bf16", "random", "tcgen05"),     # one-row tiles of 128
    (1, 1, 8, 512, 2, 256, 64, "bf16", "locality", "tcgen05"),    # 128-token pieces of tile rows
    (1, 2, 128, 8, 16, 8, 64, "bf16", "random", "tcgen05"),       # 16-row boxes
    (1, 1, 256, 2, 128, 1, 64, "bf16", "random", "tcgen05"),      # one-column tiles
    (3, 2, 48, 32, 16, 16, 64, "f32", "locality", "simt"),
]


def grid_mixing(kind, H, bh, bw, seed):
    M = bh * bw
    if kind == "locality":
        m = binding.locality_mixing(bh, bw).numpy()
        mix = np.broadcast_to(m, (H, M, M)).copy()
    else:
        u = uniform(seed, 9, (H, M, M)) + 0.05
        mix = (u / u.sum(axis=-1, keepdims=True)).astype(np.float32)
    return torch.from_numpy(mix).cuda(), mix.astype(np.float64)


@pytest.mark.parametrize("shape", GRID, ids=lambda s: "x".join(map(str, s[:7])) + f"-{s[7]}-{s[8]}")
def test_grid_blocks(shape):
    B, H, gh, gw, th, tw, d, dtype, mk, path = shape
    assert binding.mhla_forward_grid_path(B, H, gh, gw, th, tw, d, torch_dtype(dtype)) == path
    N = gh * gw
    x = rand_inputs(300 + gh + gw + d, (B, H, N, d), dtype)
    mix_t, mix64 = grid_mixing(mk, H, gh // th, gw // tw, 31 + th)
    y = torch.empty_like(x["q"])
    den = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    binding.mhla_forward_grid(x["q"], x["k"], x["v"], mix_t, y, (gh, gw), (th, tw), den_out=den)
    torch.cuda.synchronize()
    ids = oracle.grid_block_ids(gh, gw, th, tw)
    ref, dref = oracle.mhla_block_form_ids(x["q64"], x["k64"], x["v64"], mix64, ids)
    assert_close_y(to_f64(y), ref, dtype)
    assert_close_den(to_f64(den), dref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grid_of_one_row_equals_contiguous_blocks(dtype):
    """grid_h = tile_h = 1: the tiles are contiguous token ranges, the call is mhla_forward's
    (same kernel family, same arithmetic: equal bit for bit)."""
    B, H, N, d, block = 2, 3, 2048, 64, 256
    path = binding.mhla_forward_path(B, H, N, d, block, 0, torch_dtype(dtype))
    assert path == binding.mhla_forward_grid_path(B, H, 1, N, 1, block, d, torch_dtype(dtype))
    x = rand_inputs(77, (B, H, N, d), dtype)
    mix_t, _ = rand_mixing(78, H, N // block)
    y1, y2 = torch.empty_like(x["q"]), torch.empty_like(x["q"])
    binding.mhla_forward(x["q"], x["k"], x["v"], mix_t, y1, block)
    binding.mhla_forward_grid(x["q"], x["k"], x["v"], mix_t, y2, (1, N), (1, block))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_grid_tiny_brute_force():
    """A 6 x 8 grid of 2 x 4 tiles against the N x N token expansion of eq. 5."""
    B, H, gh, gw, th, tw, d = 1, 2, 6, 8, 2, 4, 16
    x = rand_inputs(91, (B, H, gh * gw, d), "f32")
    mix_t, mix64 = grid_mixing("random", H, gh // th, gw // tw, 92)
    y = torch.empty_like(x["q"])
    binding.mhla_forward_grid(x["q"], x["k"], x["v"], mix_t, y, (gh, gw), (th, tw))
    torch.cuda.synchronize()
    ref, _ = oracle.mhla_token_expansion_ids(x["q64"], x["k64"], x["v64"], mix64,
                                             oracle.grid_block_ids(gh, gw, th, tw))
    assert_close_y(to_f64(y), ref, "f32")


# ------------------------------------------------- causal MHLA inference (stream)
def lower_mixing(seed, H, M):
    """Row-normalised weights at and below the diagonal (above it: values the kernels must not read
    into the result, here large)."""
    u = np.tril(uniform(seed, 9, (H, M, M)) + 0.05)
    mix = u / u.sum(axis=-1, keepdims=True) + np.triu(np.full((M, M), 7.0), 1)
    mix = mix.astype(np.float32)
    return torch.from_numpy(mix).cuda(), np.tril(mix.astype(np.float64))


def stream_run(x, mix_t, S, z, block, t0, T, dtype):
    """Tokens t0 .. t0 + T - 1 of the [B, H, N, d] inputs through mhla_causal_stream."""
    sl = {n: x[n][:, :, t0:t0 + T].permute(2, 0, 1, 3).contiguous() for n in "qkv"}
    out = torch.empty_like(sl["q"])
    den = torch.empty(sl["q"].shape[:3], dtype=torch.float32, device="cuda")
    binding.mhla_causal_stream(sl["q"], sl["k"], sl["v"], mix_t, S, z, out, t0, block, den_out=den)
    return out, den


STREAM = [  # B, H, N, d, block, dtype
    (2, 3, 96, 16, 32, "f32"),
    (1, 2, 256, 64, 64, "bf16"),
    (1, 2, 256, 64, 64, "f32"),
    (1, 2, 128, 128, 32, "bf16"),
    (2, 1, 200, 32, 40, "f32"),
]


@pytest.mark.parametrize("shape", STREAM, ids=lambda s: "x".join(map(str, s)))
def test_causal_stream_against_the_oracle(shape):
    """Whole sequences token by token, in three calls cut inside blocks."""
    B, H, N, d, block, dtype = shape
    check_stream_calls(shape, [0, block // 2 + 1, N - block - 3, N])


# many blocks: calls that start on a block boundary and inside a block after 10 to 18 frozen
# blocks, with 1, 9, 13 and 14 blocks starting inside one call (the kernels mix the frozen
# slots of up to 8 later blocks per pass)
STREAM_MANY = [  # shape, cuts
    ((1, 2, 200, 16, 8, "f32"), [0, 80, 81, 200]),
    ((1, 2, 512, 64, 16, "bf16"), [0, 160, 300, 512]),
    ((2, 1, 384, 32, 16, "f32"), [0, 160, 163, 384]),
    ((1, 1, 256, 128, 16, "bf16"), [0, 160, 170, 256]),
]


@pytest.mark.parametrize("case", STREAM_MANY, ids=lambda c: "x".join(map(str, c[0])))
def test_causal_stream_many_blocks(case):
    check_stream_calls(*case)


def check_stream_calls(shape, cuts):
    """The sequence through one mhla_causal_stream call per range of cuts, against the oracle's
    token-by-token causal MHLA (outputs, denominators, and every block's summary slot)."""
    B, H, N, d, block, dtype = shape
    M = N // block
    x = rand_inputs(600 + N + d, (B, H, N, d), dtype)
    mix_t, mix64 = lower_mixing(601 + d, H, M)
    S = torch.full((B, H, M, d, d), float("nan"), device="cuda")  # every slot is written before it is read
    z = torch.full((B, H, M, d), float("nan"), device="cuda")
    outs, dens = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, dn = stream_run(x, mix_t, S, z, block, a, b - a, dtype)
        outs.append(o)
        dens.append(dn)
    torch.cuda.synchronize()
    y = to_f64(torch.cat(outs).permute(1, 2, 0, 3))
    den = to_f64(torch.cat(dens).permute(1, 2, 0))
    ref, dref = oracle.causal_mhla_stream(x["q64"], x["k64"], x["v64"], mix64, block)
    assert_close_y(y, ref, dtype)
    assert_close_den(den, dref, dtype)
    # the slots hold the blocks' summaries
    kf = oracle.phi(x["k64"]).reshape(B, H, M, block, d)
    s_ref = np.einsum("bhmtc,bhmte->bhmce", kf, x["v64"].reshape(B, H, M, block, d))
    assert_close_y(to_f64(S).reshape(B * H * M, 1, d, d), s_ref.reshape(B * H * M, 1, d, d), "f32",
                   what="block summaries")


def test_causal_stream_equals_the_chunk_form():
    """Token by token equals mhla_forward_causal with the same mixing and chunk = block."""
    B, H, N, d, block = 2, 2, 512, 64, 128
    M = N // block
    x = rand_inputs(640, (B, H, N, d), "bf16")
    mix_t, _ = lower_mixing(641, H, M)
    S = torch.zeros(B, H, M, d, d, device="cuda")
    z = torch.zeros(B, H, M, d, device="cuda")
    o, dn = stream_run(x, mix_t, S, z, block, 0, N, "bf16")
    yc, denc = forward_causal(x["q"], x["k"], x["v"], mix_t, block)
    torch.cuda.synchronize()
    assert slice_rel(to_f64(o.permute(1, 2, 0, 3)), yc) < 2e-2
    assert rel(to_f64(dn.permute(1, 2, 0)), denc) < 1e-4


def test_causal_stream_resumes_from_a_prefix_state():
    """The slots filled from a P-token prefix by the oracle; the next tokens give rows P.. of the
    oracle's stream over the whole sequence."""
    B, H, N, d, block, P = 1, 3, 320, 32, 64, 150
    M = N // block
    x = rand_inputs(650, (B, H, N, d), "f32")
    mix_t, mix64 = lower_mixing(651, H, M)
    kf = oracle.phi(x["k64"][:, :, :P])
    vp = x["v64"][:, :, :P]
    S0 = np.zeros((B, H, M, d, d))
    z0 = np.zeros((B, H, M, d))
    for b in range((P + block - 1) // block):
        sl = slice(b * block, min(P, (b + 1) * block))
        S0[:, :, b] = np.einsum("bhtc,bhte->bhce", kf[:, :, sl], vp[:, :, sl])
        z0[:, :, b] = kf[:, :, sl].sum(axis=2)
    S = torch.from_numpy(S0.astype(np.float32)).cuda()
    z = torch.from_numpy(z0.astype(np.float32)).cuda()
    o, dn = stream_run(x, mix_t, S, z, block, P, N - P, "f32")
    torch.cuda.synchronize()
    ref, dref = oracle.causal_mhla_stream(x["q64"], x["k64"], x["v64"], mix64, block)
    assert_close_y(to_f64(o.permute(1, 2, 0, 3)), ref[:, :, P:], "f32")
    assert_close_den(to_f64(dn.permute(1, 2, 0)), dref[:, :, P:], "f32")


def test_stream_full_workload_sampled_units():
    """The stream workload in the bench's launch configuration (4096 units, 1024 tokens after a
    2048-token prefix, M = 24): two units against the oracle over all 3072 tokens, and every
    output finite."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    runner = bench.Runner(WORKLOADS["stream"], torch.device("cuda"), 126 << 20)
    runner.step(0)
    torch.cuda.synchronize()
    s = runner.sets[0]
    assert bool(torch.isfinite(s["out"].float()).all()) and bool((s["den"] > 1e-6).all())
    res = bench.parity_of_stream(runner)
    assert res["ok"], res


# ------------------------------------------------------------ fused decode
def decode_state(seed, P, B, H, d):
    """fp32 state (S, z) summarising a P-token random prefix, and its float64 values."""
    pk = normal(seed, 1, (P, B, H, d), d ** -0.5)
    pv = normal(seed, 2, (P, B, H, d), d ** -0.5)
    kf = oracle.phi(pk)
    s0 = np.einsum("pbhc,pbhe->bhce", kf, pv).astype(np.float32)
    z0 = kf.sum(axis=0).astype(np.float32)
    return s0, z0


def decode_steps_run(S, z, q, k, v, gamma=1.0, eps=1e-6):
    out = torch.empty_like(q)
    den = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    binding.linattn_decode_steps(q, k, v, S, z, out, eps=eps, gamma=gamma, den_out=den)
    torch.cuda.synchronize()
    return to_f64(out), to_f64(den)


@pytest.mark.parametrize("gamma", [1.0, 0.9])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_decode_steps_small(d, dtype, gamma):
    """T steps in one call against the oracle's recurrence (B*H = 15 units: a
    ragged last CTA; T = 13 > the cp.async ring depth)."""
    B, H, T, P = 3, 5, 13, 40
    s0, z0 = decode_state(11 + d, P, B, H, d)
    steps = {n: rounded(normal(12 + d, 3 + i, (T, B, H, d), d ** -0.5), dtype) for i, n in enumerate("qkv")}
    S, z = torch.from_numpy(s0).cuda(), torch.from_numpy(z0).cuda()
    outs, dens = decode_steps_run(S, z, steps["q"][0], steps["k"][0], steps["v"][0], gamma)
    ref, dref, s_t, z_t = oracle.decode_steps(s0, z0, steps["q"][1], steps["k"][1], steps["v"][1], 1e-6,
                                              gamma=gamma)
    assert_close_y(outs.reshape(T * B, H, d)[:, :, None], ref.reshape(T * B, H, d)[:, :, None], dtype)
    assert_close_den(dens, dref, dtype)
    assert_close_y(to_f64(S), s_t, "f32", what="state S")
    assert rel(to_f64(z), z_t) < 1e-5


@pytest.mark.parametrize("d", [16, 64, 128])
def test_decode_steps_equal_single_steps(d):
    """gamma = 1: one fused call gives the outputs and state of T single-step calls, up to fp32
    rounding (the fused kernel's exp is the hardware base-2 exponential, about 2^-22 relative)."""
    B, H, T = 2, 7, 9
    s0, z0 = decode_state(31, 20, B, H, d)
    steps = {n: rounded(normal(32, 3 + i, (T, B, H, d), d ** -0.5), "f32")[0] for i, n in enumerate("qkv")}
    S1, z1 = torch.from_numpy(s0).cuda(), torch.from_numpy(z0).cuda()
    S2, z2 = S1.clone(), z1.clone()
    outs, dens = decode_steps_run(S1, z1, steps["q"], steps["k"], steps["v"])
    outs1, dens1 = decode_run(S2, z2, steps["q"], steps["k"], steps["v"])
    assert slice_rel(outs.reshape(T * B, H, d), outs1.reshape(T * B, H, d)) < 1e-5
    assert rel(dens, dens1) < 1e-5
    assert rel(to_f64(z1), to_f64(z2)) < 1e-5
    assert slice_rel(to_f64(S1), to_f64(S2)) < 1e-5


def test_decode_steps_zero_steps_keep_the_state():
    S = torch.randn(2, 3, 64, 64, device="cuda")
    z = torch.rand(2, 3, 64, device="cuda")
    S0, z0 = S.clone(), z.clone()
    q = torch.empty(0, 2, 3, 64, dtype=torch.bfloat16, device="cuda")
    binding.linattn_decode_steps(q, q, q, S, z, q.clone())
    torch.cuda.synchronize()
    assert torch.equal(S, S0) and torch.equal(z, z0)


def test_decode_steps_full_workload_sampled_units():
    """The decode workload's 1024 steps for all 4096 units in one call, checked
    on 65 units against the oracle; every output finite, every denominator > eps."""
    wl = WORKLOADS["decode"]
    B, H, d = wl.B, wl.H, wl.d
    dev = decode_device(wl)
    kf = torch.where(dev["prefix_k"].float() > 0, dev["prefix_k"].float() + 1, torch.exp(dev["prefix_k"].float()))
    S = torch.einsum("pbhc,pbhe->bhce", kf, dev["prefix_v"].float()).contiguous()
    z = kf.sum(dim=0).contiguous()
    units = list(range(0, B * H, 64)) + [B * H - 1]
    host = decode_host(wl, units)
    s0 = np.einsum("puc,pue->uce", oracle.phi(host["prefix_k64"]), host["prefix_v64"]).astype(np.float32)
    z0 = oracle.phi(host["prefix_k64"]).sum(axis=0).astype(np.float32)
    Sf, zf = S.view(B * H, d, d), z.view(B * H, d)
    for i, u in enumerate(units):
        Sf[u] = torch.from_numpy(s0[i]).cuda()
        zf[u] = torch.from_numpy(z0[i]).cuda()
    out = torch.empty_like(dev["step_q"])
    den = torch.empty(out.shape[:-1], dtype=torch.float32, device="cuda")
    binding.linattn_decode_steps(dev["step_q"], dev["step_k"], dev["step_v"], S, z, out, den_out=den)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out.float()).all())
    assert bool((den > 1e-6).all())
    T = wl.N
    sel = torch.tensor(units, device="cuda")
    outs = out.view(T, B * H, d)[:, sel]
    dens = den.view(T, B * H)[:, sel]
    ref, dref, s_t, z_t = oracle.decode_steps(s0, z0, host["step_q64"], host["step_k64"], host["step_v64"])
    assert_close_y(to_f64(outs).transpose(1, 0, 2)[:, None], ref.transpose(1, 0, 2)[:, None], "bf16")
    assert_close_den(to_f64(dens), dref, "bf16")
    assert_close_y(to_f64(Sf[sel])[:, None], s_t[:, None], "f32", what="state S")
    assert rel(to_f64(zf[sel]), z_t) < 1e-5


# ----------------------------------------------------------------------- RALA
RALA = [  # B, H, N, d, cx
    (2, 2, 200, 16, 32),
    (1, 2, 256, 32, 64),
    (2, 1, 600, 64, 16),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", RALA, ids=lambda s: "x".join(map(str, s)))
def test_rala_small(shape, dtype):
    B, H, N, d, cx = shape
    x = rand_inputs(300 + N, (B, H, N, d), dtype)
    xt, x64 = rounded(normal(301, 5, (B, N, cx)), dtype)
    wt, w64 = rounded(normal(301, 6, (cx, d), cx ** -0.5), dtype)
    y = torch.empty_like(x["q"])
    binding.rala_forward(x["q"], x["k"], x["v"], xt, wt, y)
    torch.cuda.synchronize()
    ref = oracle.rala_forward(x["q64"], x["k64"], x["v64"], x64, w64)
    assert_close_y(to_f64(y), ref, dtype)


# bf16, d = 32, Cx = 64, H <= 2, N a multiple of 64: the tensor-core RALA
# kernels (token pairs as 128-byte rows, tiles of 128 pairs).  The offset on
# Q moves Q_g away from zero, so the logits span tens of units and the
# softmax depends on its maximum being taken out first.
RALA_TC = [  # B, H, N, q offset
    (3, 2, 832, 0.0),     # 416 pairs: three whole tiles and a quarter tile
    (2, 1, 1024, 0.0),    # one head, whole tiles only
    (1, 2, 64, 0.0),      # a single quarter-filled tile
    (2, 2, 448, 1.5),     # peaked softmax
]


@pytest.mark.parametrize("shape", RALA_TC, ids=lambda s: "x".join(map(str, s)))
def test_rala_tcgen05_shapes(shape):
    B, H, N, off = shape
    d, cx = 32, 64
    q64 = normal(310 + N, 1, (B, H, N, d), d ** -0.5) + off
    qt, q64 = rounded(q64, "bf16")
    x = rand_inputs(310 + N, (B, H, N, d), "bf16")
    xt, x64 = rounded(normal(311, 5, (B, N, cx)), "bf16")
    wt, w64 = rounded(normal(311, 6, (cx, d), cx ** -0.5), "bf16")
    y = torch.empty_like(qt)
    binding.rala_forward(qt, x["k"], x["v"], xt, wt, y)
    torch.cuda.synchronize()
    ref = oracle.rala_forward(q64, x["k64"], x["v64"], x64, w64)
    assert_close_y(to_f64(y), ref, "bf16")


def test_rala_full_workload_every_batch():
    wl = WORKLOADS["rala"]
    dev = rala_device(wl)
    y = torch.empty_like(dev["q"])
    binding.rala_forward(dev["q"], dev["k"], dev["v"], dev["x"], dev["w"], y)
    torch.cuda.synchronize()
    y = to_f64(y)
    assert np.all(np.isfinite(y))
    batches = list(range(wl.B))
    host = rala_host(wl, batches)
    ref = oracle.rala_forward(host["q64"], host["k64"], host["v64"], host["x64"], host["w64"])
    assert_close_y(y[batches], ref, wl.dtype)
