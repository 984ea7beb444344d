"""GPU parity of the MHLA backward (dQ, dK, dV, dM) through the C ABI against the float64 oracle.

The oracle's backward is pinned to its forward by central differences (tests/test_oracle_pins.py).
Tolerances, relative to the largest magnitude of each gradient tensor: fp32 1e-4 (the kernels
sum in fp32 over at most a block of tokens or d features); bf16 gradients 1e-2 (each is rounded
once to bf16, 2^-9 relative, on top of the fp32 sums).  dM is fp32 in both dtypes and is a sum of
B (d^2 + d) products <dS~_i, S_b> + dz~_i . z_b whose terms can nearly cancel (Euler's identity
makes sum_b m_ib dm_ib vanish as eps -> 0), so its bound adds 1e-5 times the sum of the terms'
magnitudes (fp32 rounding of the summed terms and of dS~, S themselves) to 1e-3 of max |dM|.
The tensor-core path (bf16, d = 64, blocks of whole 128-token chunks) multiplies bf16 operands
(phi(Q), phi(K), V, dY, dnum, dden and the bf16-rounded S~, dS: 2^-9 each, two per product, and
dden inherits the bf16 products of num): its gradients are held to 2e-2, the forward's bf16 bound,
and dM to 2^-6 times the absolute products summed inside dS~ and dz~, times |S|, |z|.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import to_f64, torch_dtype
from test_parity_gpu import rand_inputs, rand_mixing, rounded
from token_level_head_gb300 import binding
from token_level_head_gb300.build import build_library
from workloads import WORKLOADS, mhla_device, mhla_host, normal

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2, "tcgen05": 2e-2}
TOL_DM, TOL_DM_TERMS, TOL_DM_TC = 1e-3, 1e-5, 2.0 ** -6


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_library()
    return binding.load()


def rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def backward(q, k, v, mix, dy, block, eps=1e-6):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dm = torch.empty_like(mix)
    binding.mhla_backward(q, k, v, mix, dy, dq, dk, dv, dm, block, eps=eps)
    torch.cuda.synchronize()
    return to_f64(dq), to_f64(dk), to_f64(dv), to_f64(dm)


def dm_term_magnitudes(q, k, v, mix, block, dy, eps, absolute=False):
    """sum over samples and entries of |dS~_i| |S_b| + |dz~_i| |z_b|, [H, M, M] (float64): the scale of
    the cancelling sum that gives dm_ib.  absolute: dS~ and dz~ replaced by the sums of the absolute
    values of their products (sum_t |phi(q_t)| |dnum_t|, and |dden_t| plus the spread of num's
    products sum_e |dY_e| sum_c |phi_c| |S~_ce| / den^2), the scale of bf16 operand rounding."""
    B, H, N, d = q.shape
    M = N // block
    kf = oracle.phi(k).reshape(B, H, M, block, d)
    s = np.einsum("bhmjc,bhmje->bhmce", kf, v.reshape(B, H, M, block, d))
    z = kf.sum(axis=3)
    s_mix, z_mix = np.einsum("hib,zhbce->zhice", mix, s), np.einsum("hib,zhbc->zhic", mix, z)
    qf = oracle.phi(q).reshape(B, H, M, block, d)
    g = dy.reshape(B, H, M, block, d)
    num = np.einsum("bhitc,bhice->bhite", qf, s_mix)
    den = np.einsum("bhitc,bhic->bhit", qf, z_mix) + eps
    dden = -np.einsum("bhite,bhite->bhit", g, num) / den ** 2
    ds_mix = np.einsum("bhitc,bhite->bhice", qf, g / den[..., None])
    dz_mix = np.einsum("bhitc,bhit->bhic", qf, dden)
    if absolute:
        ds_mix = np.einsum("bhitc,bhite->bhice", np.abs(qf), np.abs(g) / den[..., None])
        spread = np.einsum("bhite,bhitc,bhice->bhit", np.abs(g), np.abs(qf), np.abs(s_mix)) / den ** 2
        dz_mix = np.einsum("bhitc,bhit->bhic", np.abs(qf), np.abs(dden) + spread)
    return (np.einsum("zhice,zhbce->hib", np.abs(ds_mix), np.abs(s))
            + np.einsum("zhic,zhbc->hib", np.abs(dz_mix), np.abs(z)))


def check(got, ref, dtype, terms=None, path="simt"):
    """terms: dm_term_magnitudes of the case (absolute=True on the tensor-core path)."""
    tol = TOL["tcgen05"] if path == "tcgen05" else TOL[dtype]
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        assert rel_err(g, r) <= tol, (name, rel_err(g, r))
    scale = TOL_DM_TC if path == "tcgen05" else TOL_DM_TERMS
    bound = TOL_DM * np.max(np.abs(ref[3])) + (0.0 if terms is None else scale * terms)
    assert np.all(np.abs(got[3] - ref[3]) <= bound), ("dmixing", rel_err(got[3], ref[3]))


def checked(inp, mix_dev, mix_host, dy, dy64, block, dtype, eps=1e-6):
    """The backward of these inputs against the oracle, with the bound of the path it runs."""
    B, H, N, d = inp["q64"].shape
    path = binding.mhla_backward_path(B, H, N, d, block, torch_dtype(dtype))
    args = (inp["q64"], inp["k64"], inp["v64"], mix_host, block, dy64, eps)
    got = backward(inp["q"], inp["k"], inp["v"], mix_dev, dy, block, eps)
    check(got, oracle.mhla_block_form_backward(*args), dtype,
          dm_term_magnitudes(*args, absolute=path == "tcgen05"), path)
    return path


BWD = [  # B, H, N, d, block, dtype, eps
    (2, 3, 256, 64, 64, "f32", 1e-6),
    (2, 3, 512, 64, 128, "f32", 1e-6),    # fp32: the SIMT passes at a tensor-core shape
    (1, 2, 200, 32, 40, "f32", 1e-6),     # blocks shorter than a chunk of 64 tokens
    (1, 2, 384, 16, 96, "f32", 1e-6),     # a full chunk and a ragged one per block
    (1, 1, 256, 128, 64, "f32", 1e-6),    # d = 128: chunks of 32 tokens
    (2, 2, 512, 64, 128, "bf16", 1e-6),
    (1, 2, 1024, 64, 16, "bf16", 1e-6),   # M = 64, the most blocks
    # M = 1, global linear attention: Y depends on the single weight only through eps (dM = 0 in
    # exact arithmetic when eps = 0), so a large eps gives dM a value to compare
    (3, 2, 320, 32, 320, "bf16", 0.5),
    (2, 1, 192, 128, 96, "bf16", 1e-6),
    # tensor-core token passes: blocks of one and of three chunks, M = 1 and M = 32
    (1, 3, 768, 64, 384, "bf16", 1e-6),
    (3, 1, 256, 64, 256, "bf16", 0.5),
    (1, 2, 4096, 64, 128, "bf16", 1e-6),
]


@pytest.mark.parametrize("shape", BWD, ids=lambda s: "x".join(map(str, s[:6])))
def test_backward_against_the_oracle(shape):
    B, H, N, d, block, dtype, eps = shape
    x = rand_inputs(900 + N + d, (B, H, N, d), dtype)
    dy, dy64 = rounded(normal(901 + N, 4, (B, H, N, d)), dtype)
    mix_t, mix64 = rand_mixing(902 + block, H, N // block)
    path = checked(x, mix_t, mix64, dy, dy64, block, dtype, eps)
    assert path == ("tcgen05" if dtype == "bf16" and d == 64 and block % 128 == 0 else "simt")


@pytest.mark.parametrize("dtype,block", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_backward_edge_cases(dtype, block):
    """eps = 0; inputs of std 1 instead of d^-1/2 (phi far into both branches); identity mixing
    (blockwise linear attention; dM off the diagonal still nonzero); exact zeros in the mixing.
    bf16 with blocks of 128 runs the tensor-core passes, the others the SIMT ones."""
    B, H, N, d = 2, 2, 512, 64
    M = N // block
    dy, dy64 = rounded(normal(911, 4, (B, H, N, d)), dtype)
    x = rand_inputs(910, (B, H, N, d), dtype)
    mix_t, mix64 = rand_mixing(912, H, M)

    def case(inp, mix_dev, mix_host, eps=1e-6):
        checked(inp, mix_dev, mix_host, dy, dy64, block, dtype, eps)

    case(x, mix_t, mix64, eps=0.0)
    case(rand_inputs(913, (B, H, N, d), dtype, scale=1.0), mix_t, mix64)
    eye = np.ascontiguousarray(np.broadcast_to(np.eye(M), (H, M, M)))
    case(x, torch.from_numpy(eye.astype(np.float32)).cuda(), eye)
    holes = mix64 * (np.arange(M)[None, :, None] != np.arange(M)[None, None, :] + 1)  # zero subdiagonal
    case(x, torch.from_numpy(holes.astype(np.float32)).cuda(), holes)


def test_backward_is_deterministic():
    B, H, N, d, block = 2, 3, 512, 64, 128
    x = rand_inputs(920, (B, H, N, d), "bf16")
    dy, _ = rounded(normal(921, 4, (B, H, N, d)), "bf16")
    mix_t, _ = rand_mixing(922, H, N // block)
    a = backward(x["q"], x["k"], x["v"], mix_t, dy, block)
    b = backward(x["q"], x["k"], x["v"], mix_t, dy, block)
    assert all(np.array_equal(p, r) for p, r in zip(a, b))


def test_backward_full_workload_sampled_heads():
    """The DiT backward workload (B8 H6 N4096 d64, M = 16, bf16) as the bench runs it: every output
    finite; all eight samples of heads 0 and 5 (their dQ, dK, dV and the whole dM row of the head)
    against the oracle."""
    wl = WORKLOADS["dit_backward"]
    dev = mhla_device(wl)
    got = backward(dev["q"], dev["k"], dev["v"], dev["mixing"], dev["dy"], wl.block)
    for g in got:
        assert np.isfinite(g).all()
    for h in (0, wl.H - 1):
        host = mhla_host(wl, heads=[(b, h) for b in range(wl.B)])
        shp = (wl.B, 1, wl.N, wl.d)
        args = (host["q64"].reshape(shp), host["k64"].reshape(shp), host["v64"].reshape(shp),
                host["mixing64"][:1], wl.block, host["dy64"].reshape(shp), 1e-6)
        sub = tuple(g[:, h:h + 1] for g in got[:3]) + (got[3][h:h + 1],)
        check(sub, oracle.mhla_block_form_backward(*args), "bf16", dm_term_magnitudes(*args, absolute=True),
              "tcgen05")
    assert binding.mhla_backward_path(wl.B, wl.H, wl.N, wl.d, wl.block, torch.bfloat16) == "tcgen05"
