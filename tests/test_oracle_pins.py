"""Pins of the CPU oracle to things other than itself.

Each test fixes an oracle function against a hand-derived fixture, a closed
form, an invariant stated by the source pages, or a second, differently
written definition (block form against token expansion, recurrence against
chunked form against masked brute force).  These run on the CPU only.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, mhla_host, normal, uniform

TOL = 1e-12


def close(a, b, tol=TOL):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return a.shape == b.shape and float(np.max(np.abs(a - b))) <= tol * scale


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def as4(x):
    """[N, d] fixture array -> [1, 1, N, d]."""
    return np.asarray(x, dtype=np.float64)[None, None]


# ---------------------------------------------------------------- phi
def test_phi_closed_forms():
    assert oracle.phi(0.0) == 1.0
    assert oracle.phi(1.0) == 2.0
    assert oracle.phi(2.5) == 3.5
    assert math.isclose(oracle.phi(-1.0), math.exp(-1.0), rel_tol=0, abs_tol=1e-16)
    assert math.isclose(oracle.phi(-math.log(2.0)), 0.5, rel_tol=1e-15)
    assert oracle.phi(-800.0) == 0.0
    # continuity at 0 and positivity everywhere (a positive feature map, Linear Attention notes §二)
    assert abs(oracle.phi(1e-12) - oracle.phi(-1e-12)) < 1e-11
    x = np.linspace(-30, 30, 10001)
    assert np.all(oracle.phi(x) > 0)
    assert np.all(np.diff(oracle.phi(x)) > 0)


# ------------------------------------------------------- golden fixtures
def test_golden_linear_attention(golden_dir):
    for name in ("linear_attention_d1.json", "linear_attention_d2_eps.json"):
        fx = load(golden_dir, name)
        q, k, v, eps = as4(fx["q"]), as4(fx["k"]), as4(fx["v"]), fx["eps"]
        n = q.shape[2]
        y, den = oracle.global_linear_attention(q, k, v, eps)
        assert close(y[0, 0], fx["noncausal_y"]) and close(den[0, 0], fx["noncausal_den"]), name
        one = np.ones((1, 1, 1))
        y, den = oracle.mhla_block_form(q, k, v, one, n, eps)
        assert close(y[0, 0], fx["noncausal_y"]) and close(den[0, 0], fx["noncausal_den"]), name
        y, den = oracle.mhla_token_expansion(q, k, v, one, n, eps)
        assert close(y[0, 0], fx["noncausal_y"]) and close(den[0, 0], fx["noncausal_den"]), name
        for fn in (oracle.causal_recurrent, oracle.causal_bruteforce):
            y, den = fn(q, k, v, eps)
            assert close(y[0, 0], fx["causal_y"]) and close(den[0, 0], fx["causal_den"]), (name, fn)
        y, den = oracle.causal_chunked(q, k, v, 1, eps)
        assert close(y[0, 0], fx["causal_y"]) and close(den[0, 0], fx["causal_den"]), name
        # decode: one prefix token, then one step
        s0 = oracle.phi(k[0, 0, 0])[:, None] * v[0, 0, 0][None, :]
        outs, dens, _, _ = oracle.decode_steps(s0, oracle.phi(k[0, 0, 0]), q[0, 0, 1:], k[0, 0, 1:],
                                               v[0, 0, 1:], eps)
        assert close(outs[0], fx["causal_y"][1]) and close(dens[0], fx["causal_den"][1]), name


def test_golden_mhla_two_blocks(golden_dir):
    fx = load(golden_dir, "mhla_two_blocks_d1.json")
    q, k, v, eps = as4(fx["q"]), as4(fx["k"]), as4(fx["v"]), fx["eps"]
    mix = np.asarray(fx["mixing"])[None]
    for fn in (oracle.mhla_block_form, oracle.mhla_token_expansion):
        y, den = fn(q, k, v, mix, fx["block_size"], eps)
        assert close(y[0, 0], fx["noncausal_y"]) and close(den[0, 0], fx["noncausal_den"]), fn
    for fn in (oracle.causal_mhla_chunked, oracle.causal_mhla_bruteforce):
        y, den = fn(q, k, v, mix, fx["block_size"], eps)
        assert close(y[0, 0], fx["causal_y"]) and close(den[0, 0], fx["causal_den"]), fn


def test_golden_rala(golden_dir):
    fx = load(golden_dir, "rala_d1.json")
    q, k, v = as4(fx["q"]), as4(fx["k"]), as4(fx["v"])
    x, w = np.asarray(fx["x"])[None], np.asarray(fx["w"])
    for fn in (oracle.rala_forward, oracle.rala_bruteforce):
        assert close(fn(q, k, v, x, w)[0, 0], fx["y"]), fn


# ------------------------------------------- two definitions of MHLA agree
@pytest.fixture(scope="module")
def tiny():
    wl = WORKLOADS["tiny"]
    return wl, mhla_host(wl)


def test_block_form_equals_token_expansion_tiny(tiny):
    wl, x = tiny
    y1, d1 = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block, 1e-6)
    y2, d2 = oracle.mhla_token_expansion(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block, 1e-6)
    assert close(y1, y2, 1e-11) and close(d1, d2, 1e-11)
    # the tiny workload's mixing is genuinely asymmetric, so a transposed m is caught here
    assert np.max(np.abs(x["mixing64"][0] - x["mixing64"][0].T)) > 0.05


def test_closed_form_constant_features():
    """Q = K = 0 gives phi = 1, so every score is d and Y_t is a mixed block mean of V.

    Y_t = d * sum_b m_{i,b} sum_{s in b} v_s / (d * sum_b m_{i,b} n_b + eps),
    written here from block sums of V alone (no phi, S or z).
    """
    n, d, nb, eps = 48, 3, 12, 0.37
    m = n // nb
    v = normal(7, 1, (1, 2, n, d))
    mix = uniform(7, 2, (2, m, m)) + 0.1
    zero = np.zeros_like(v)
    block_sums = v.reshape(1, 2, m, nb, d).sum(axis=3)            # [1, 2, M, d]
    expect = np.empty_like(v)
    for h in range(2):
        for t in range(n):
            i = t // nb
            num = d * (mix[h, i][:, None] * block_sums[0, h]).sum(axis=0)
            expect[0, h, t] = num / (d * mix[h, i].sum() * nb + eps)
    for fn in (oracle.mhla_block_form, oracle.mhla_token_expansion):
        y, _ = fn(zero, zero, v, mix, nb, eps)
        assert close(y, expect, 1e-12), fn


def test_m1_and_all_ones_mixing_equal_global_linear_attention(tiny):
    wl, x = tiny
    q, k, v = x["q64"], x["k64"], x["v64"]
    ref, dref = oracle.global_linear_attention(q, k, v, 1e-6)
    y, den = oracle.mhla_block_form(q, k, v, np.ones((1, 1, 1)), wl.N, 1e-6)
    assert close(y, ref, 1e-12) and close(den, dref, 1e-12)
    y, den = oracle.mhla_block_form(q, k, v, np.ones((1, wl.M, wl.M)), wl.block, 1e-6)
    assert close(y, ref, 1e-12) and close(den, dref, 1e-12)


def test_identity_mixing_is_blockwise_linear_attention(tiny):
    wl, x = tiny
    q, k, v = x["q64"], x["k64"], x["v64"]
    y, _ = oracle.mhla_block_form(q, k, v, np.eye(wl.M)[None], wl.block, 1e-6)
    for b in range(wl.M):
        sl = slice(b * wl.block, (b + 1) * wl.block)
        ref, _ = oracle.global_linear_attention(q[..., sl, :], k[..., sl, :], v[..., sl, :], 1e-6)
        assert close(y[..., sl, :], ref, 1e-12)


def test_row_scaling_of_mixing_leaves_output_unchanged(tiny):
    """The output is a ratio (MHLA paper §4.1), so scaling row i of m by c > 0 cancels when eps = 0."""
    wl, x = tiny
    q, k, v, mix = x["q64"], x["k64"], x["v64"], x["mixing64"]
    scaled = mix * np.array([0.5, 3.0, 7.0, 0.01])[None, :, None]
    y1, _ = oracle.mhla_block_form(q, k, v, mix, wl.block, 0.0)
    y2, _ = oracle.mhla_block_form(q, k, v, scaled, wl.block, 0.0)
    assert close(y1, y2, 1e-12)


def test_permutation_inside_a_block(tiny):
    """Summaries are sums over a block, so permuting the tokens of block 1 permutes only block 1's outputs."""
    wl, x = tiny
    q, k, v, mix = x["q64"], x["k64"], x["v64"], x["mixing64"]
    perm = np.arange(wl.N)
    sl = np.arange(wl.block, 2 * wl.block)
    perm[sl] = sl[::-1]
    y1, _ = oracle.mhla_block_form(q, k, v, mix, wl.block, 1e-6)
    y2, _ = oracle.mhla_block_form(q[..., perm, :], k[..., perm, :], v[..., perm, :], mix, wl.block, 1e-6)
    assert close(y2, y1[..., perm, :], 1e-12)


# ------------------------------------------------------------- rank pins
def test_rank_of_linear_attention_matrix_is_at_most_d(tiny):
    """MHLA paper §3.2: rank(phi(Q) phi(K)^T) <= d whatever N is."""
    wl, x = tiny
    a = oracle.mhla_attention_matrix(x["q64"][0, 0], x["k64"][0, 0], np.ones((wl.M, wl.M)), wl.block)
    assert a.shape == (wl.N, wl.N)
    assert oracle.numerical_rank(a) == wl.d


def test_rank_of_mhla_matrix_reaches_sum_of_block_ranks(tiny):
    """MHLA paper §4.3: rank(A_MHLA) <= min(n, sum_b min(n_b, d)), attained for generic mixing."""
    wl, x = tiny
    a = oracle.mhla_attention_matrix(x["q64"][0, 0], x["k64"][0, 0], x["mixing64"][0], wl.block)
    bound = min(wl.N, wl.M * min(wl.block, wl.d))
    assert bound == 64
    assert oracle.numerical_rank(a) == bound


def test_numerical_rank_on_known_matrices():
    assert oracle.numerical_rank(np.diag([3.0, 2.0, 1.0, 0.0, 0.0])) == 3
    assert oracle.numerical_rank(np.zeros((4, 4))) == 0
    assert oracle.numerical_rank(np.outer(np.arange(1, 6), np.arange(1, 4))) == 1


# ----------------------------------------------------------- causal pins
@pytest.fixture(scope="module")
def causal_small():
    q = normal(11, 1, (2, 2, 96, 8), 0.4)
    k = normal(11, 2, (2, 2, 96, 8), 0.4)
    v = normal(11, 3, (2, 2, 96, 8))
    return q, k, v


def test_causal_three_ways(causal_small):
    q, k, v = causal_small
    ref, dref = oracle.causal_bruteforce(q, k, v, 1e-6)
    y, den = oracle.causal_recurrent(q, k, v, 1e-6)
    assert close(y, ref, 1e-11) and close(den, dref, 1e-11)
    for c in (1, 16, 32, 96, 40):        # 40: ragged last chunk
        y, den = oracle.causal_chunked(q, k, v, c, 1e-6)
        assert close(y, ref, 1e-11) and close(den, dref, 1e-11), c


def test_causal_last_token_sees_everything(causal_small):
    q, k, v = causal_small
    y, den = oracle.causal_recurrent(q, k, v, 1e-6)
    g, dg = oracle.global_linear_attention(q, k, v, 1e-6)
    assert close(y[..., -1, :], g[..., -1, :], 1e-12) and close(den[..., -1], dg[..., -1], 1e-12)


def test_causal_mhla_chunked_equals_bruteforce(causal_small):
    q, k, v = causal_small
    mix = np.tril(uniform(3, 4, (2, 4, 4)) + 0.05)
    y1, d1 = oracle.causal_mhla_chunked(q, k, v, mix, 24, 1e-6)
    y2, d2 = oracle.causal_mhla_bruteforce(q, k, v, mix, 24, 1e-6)
    assert close(y1, y2, 1e-11) and close(d1, d2, 1e-11)
    # entries above the diagonal are ignored
    y3, _ = oracle.causal_mhla_chunked(q, k, v, mix + np.triu(np.ones((4, 4)), 1)[None], 24, 1e-6)
    assert close(y3, y1, 1e-12)


def test_causal_mhla_all_ones_is_causal_linear_attention(causal_small):
    q, k, v = causal_small
    ref, dref = oracle.causal_recurrent(q, k, v, 1e-6)
    for fn in (oracle.causal_mhla_chunked, oracle.causal_mhla_bruteforce):
        y, den = fn(q, k, v, np.ones((2, 4, 4)), 24, 1e-6)
        assert close(y, ref, 1e-11) and close(den, dref, 1e-11), fn


def test_decode_continues_the_causal_sequence(causal_small):
    """P prefix tokens then T decode steps give rows P..P+T-1 of the causal forward."""
    q, k, v = causal_small
    p = 64
    ref, dref = oracle.causal_bruteforce(q, k, v, 1e-6)
    kf = oracle.phi(k[..., :p, :])
    s0 = np.einsum("bhjc,bhje->bhce", kf, v[..., :p, :])
    z0 = kf.sum(axis=2)
    steps = lambda x: np.moveaxis(x[..., p:, :], 2, 0)  # noqa: E731  [T, B, H, d]
    outs, dens, s_t, z_t = oracle.decode_steps(s0, z0, steps(q), steps(k), steps(v), 1e-6)
    assert close(np.moveaxis(outs, 0, 2), ref[..., p:, :], 1e-11)
    assert close(np.moveaxis(dens, 0, 2), dref[..., p:], 1e-11)
    # the final state is the summary of the whole sequence, as the block form computes it
    whole = oracle.mhla_block_form(q, k, v, np.ones((2, 1, 1)), 96, 1e-6)[1]
    assert close(np.einsum("bhtc,bhc->bht", oracle.phi(q), z_t) + 1e-6, whole, 1e-12)


# ------------------------------------------------------------- RALA pins
@pytest.fixture(scope="module")
def rala_small():
    q = normal(5, 1, (2, 2, 40, 8), 8 ** -0.5)
    k = normal(5, 2, (2, 2, 40, 8), 8 ** -0.5)
    v = normal(5, 3, (2, 2, 40, 8), 8 ** -0.5)
    x = normal(5, 5, (2, 40, 16))
    w = normal(5, 6, (16, 8), 0.25)
    return q, k, v, x, w


def test_rala_forward_equals_bruteforce(rala_small):
    q, k, v, x, w = rala_small
    assert close(oracle.rala_forward(q, k, v, x, w), oracle.rala_bruteforce(q, k, v, x, w), 1e-11)


def test_rala_zero_queries_weight_all_keys_equally(rala_small):
    """Q = 0 gives Q_g = 0, so alpha_j = 1/N and phi(Q) = 1: Y_t = (XW)_t * mean_s (sum_c phi(k_s)_c) v_s."""
    _, k, v, x, w = rala_small
    q = np.zeros_like(k)
    y = oracle.rala_forward(q, k, v, x, w)
    ksum = oracle.phi(k).sum(axis=-1)                                  # [B, H, N]
    mean = (ksum[..., None] * v).mean(axis=2)                          # [B, H, d]
    expect = np.einsum("bnc,cd->bnd", x, w)[:, None] * mean[:, :, None, :]
    assert close(y, expect, 1e-12)


def test_rala_zero_keys_give_mean_value(rala_small):
    """K = 0 gives phi(K) = 1 and equal logits, so B has every row equal to mean(V)."""
    q, _, v, x, w = rala_small
    k = np.zeros_like(q)
    y = oracle.rala_bruteforce(q, k, v, x, w)
    qsum = oracle.phi(q).sum(axis=-1)                                  # [B, H, N]
    expect = np.einsum("bnc,cd->bnd", x, w)[:, None] * (qsum[..., None] * v.mean(axis=2)[:, :, None, :])
    assert close(y, expect, 1e-12)


def test_rala_one_dominant_key(rala_small):
    """One key far above the rest takes all the softmax weight: B = phi(k*) v*^T, so with Q = 1
    (phi(Q) = 2) Y_t = (XW)_t * 2 d (1 + 30) v*."""
    _, _, v, x, w = rala_small
    q = np.ones_like(v)
    k = np.zeros_like(v)
    k[..., 7, :] = 30.0
    d = v.shape[-1]
    expect = np.einsum("bnc,cd->bnd", x, w)[:, None] * (2.0 * d * 31.0 * v[..., 7, :])[:, :, None, :]
    for fn in (oracle.rala_forward, oracle.rala_bruteforce):
        assert close(fn(q, k, v, x, w), expect, 1e-12), fn


# --------------------------------------------------- decay (RetNet) pins
def test_decayed_bruteforce_special_cases(causal_small):
    q, k, v = causal_small
    ref, dref = oracle.causal_bruteforce(q, k, v, 1e-6)
    y1, d1 = oracle.decayed_causal_bruteforce(q, k, v, 1.0, 1e-6)
    assert close(y1, ref, 1e-12) and close(d1, dref, 1e-12)
    # gamma = 0: every token sees only itself, so out_t = v_t (eps negligible)
    y0, d0 = oracle.decayed_causal_bruteforce(q, k, v, 0.0, 0.0)
    assert close(y0, v, 1e-12)
    assert close(d0, np.einsum("...tc,...tc->...t", oracle.phi(q), oracle.phi(k)), 1e-12)


def test_decayed_bruteforce_two_tokens_by_hand():
    """d = 1, tokens x = [0, ln 2]: phi = [1, 3];  gamma = 1/2, v = [2, 5], q = [0, 0] (phi 1):
    out_0 = 1*2 / 1 = 2;  out_1 = (0.5 * 1 * 2 + 1 * 3 * 5) / (0.5 * 1 + 3) = 16 / 3.5."""
    q = np.zeros((1, 1, 2, 1))
    k = np.array([0.0, math.log(2.0)]).reshape(1, 1, 2, 1)
    k[0, 0, 1, 0] = 2.0  # phi(2) = 3
    v = np.array([2.0, 5.0]).reshape(1, 1, 2, 1)
    y, den = oracle.decayed_causal_bruteforce(q, k, v, 0.5, 0.0)
    assert close(y.ravel(), [2.0, 16.0 / 3.5], 1e-14) and close(den.ravel(), [1.0, 3.5], 1e-14)


def test_decode_with_decay_equals_decayed_bruteforce(causal_small):
    q, k, v = causal_small
    s0 = normal(12, 1, (2, 2, 8, 8))
    z0 = np.abs(normal(12, 2, (2, 2, 8))) + 1.0
    steps = lambda x: np.moveaxis(x, 2, 0)  # noqa: E731  [T, B, H, d]
    for gamma in (0.9, 0.5):
        outs, dens, s_t, z_t = oracle.decode_steps(s0, z0, steps(q), steps(k), steps(v), 1e-6, gamma=gamma)
        ref, dref = oracle.decayed_causal_bruteforce(q, k, v, gamma, 1e-6, s0=s0, z0=z0)
        assert close(np.moveaxis(outs, 0, 2), ref, 1e-10) and close(np.moveaxis(dens, 0, 2), dref, 1e-10)
        n = q.shape[2]
        w = gamma ** np.arange(n - 1, -1, -1)
        s_ref = gamma ** n * s0 + np.einsum("t,bhtc,bhte->bhce", w, oracle.phi(k), v)
        assert close(s_t, s_ref, 1e-10)


# ------------------------------------------------- normaliser-free pins
def test_unnormalized_equals_bruteforce_sum(tiny):
    wl, x = tiny
    mix, block = x["mixing64"], wl.block
    num = oracle.mhla_block_form_unnormalized(x["q64"], x["k64"], x["v64"], mix, block)
    a = oracle.mhla_attention_matrix(x["q64"][0, 0], x["k64"][0, 0], mix[0], block)
    assert close(num[0, 0], a @ x["v64"][0, 0], 1e-11)
    y, den = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], mix, block, 1e-6)
    assert close(num, y * den[..., None], 1e-11)


# ---------------------------------------------------- 2-D block pins
def test_grid_block_ids_by_hand():
    ids = oracle.grid_block_ids(4, 4, 2, 2)
    assert ids.tolist() == [0, 0, 1, 1, 0, 0, 1, 1, 2, 2, 3, 3, 2, 2, 3, 3]
    assert oracle.grid_block_ids(2, 6, 1, 6).tolist() == [0] * 6 + [1] * 6


@pytest.fixture(scope="module")
def grid_small():
    q = normal(21, 1, (1, 2, 64, 4), 0.5)   # an 8 x 8 token grid
    k = normal(21, 2, (1, 2, 64, 4), 0.5)
    v = normal(21, 3, (1, 2, 64, 4))
    u = uniform(21, 4, (2, 4, 4)) + 0.05
    return q, k, v, u / u.sum(axis=-1, keepdims=True)


def test_grid_blocks_equal_token_expansion(grid_small):
    q, k, v, mix = grid_small
    ids = oracle.grid_block_ids(8, 8, 4, 4)
    y1, d1 = oracle.mhla_block_form_ids(q, k, v, mix, ids, 1e-6)
    y2, d2 = oracle.mhla_token_expansion_ids(q, k, v, mix, ids, 1e-6)
    assert close(y1, y2, 1e-11) and close(d1, d2, 1e-11)


def test_contiguous_ids_equal_the_1d_block_form(grid_small):
    q, k, v, mix = grid_small
    ids = oracle.block_of(64, 16)
    y1, d1 = oracle.mhla_block_form_ids(q, k, v, mix, ids, 1e-6)
    y2, d2 = oracle.mhla_block_form(q, k, v, mix, 16, 1e-6)
    assert close(y1, y2, 1e-12) and close(d1, d2, 1e-12)
    y3, d3 = oracle.mhla_token_expansion_ids(q, k, v, mix, ids, 1e-6)
    y4, d4 = oracle.mhla_token_expansion(q, k, v, mix, 16, 1e-6)
    assert close(y3, y4, 1e-12) and close(d3, d4, 1e-12)
    # rows of the grid as tiles (tile_h = 1... here 2 rows of 8 = 16 tokens) are contiguous blocks
    assert oracle.grid_block_ids(8, 8, 2, 8).tolist() == ids.tolist()


def test_grid_blocks_are_1d_blocks_of_the_tile_ordered_tokens(grid_small):
    q, k, v, mix = grid_small
    ids = oracle.grid_block_ids(8, 8, 4, 4)
    order = np.argsort(ids, kind="stable")   # tokens of tile 0, then tile 1, ...
    y1, d1 = oracle.mhla_block_form_ids(q, k, v, mix, ids, 1e-6)
    y2, d2 = oracle.mhla_block_form(q[:, :, order], k[:, :, order], v[:, :, order], mix, 16, 1e-6)
    assert close(y1[:, :, order], y2, 1e-12) and close(d1[:, :, order], d2, 1e-12)


def test_locality_init_by_hand():
    m = oracle.locality_mixing_init(1, 3)
    assert close(m, [[2 / 3, 1 / 3, 0], [0, 1, 0], [0, 1 / 3, 2 / 3]], 1e-15)
    m = oracle.locality_mixing_init(2, 2)
    a = 1 - 1 / math.sqrt(2)
    row0 = np.array([1, a, a, 0]) / (1 + 2 * a)
    assert close(m[0], row0, 1e-15) and close(m[3], row0[::-1], 1e-15)
    assert close(oracle.locality_mixing_init(1, 1), [[1.0]], 0)
    m = oracle.locality_mixing_init(5, 5)       # Fig. 4b's M = 25
    assert close(m.sum(axis=1), np.ones(25), 1e-14) and np.all(m >= 0)
    assert np.all(np.argmax(m, axis=1) == np.arange(25))


# ------------------------------------------- streaming causal MHLA pins
def test_causal_mhla_stream_equals_bruteforce(causal_small):
    q, k, v = causal_small
    mix = np.tril(uniform(5, 4, (2, 4, 4)) + 0.05)
    y1, d1 = oracle.causal_mhla_stream(q, k, v, mix, 24, 1e-6)
    y2, d2 = oracle.causal_mhla_bruteforce(q, k, v, mix, 24, 1e-6)
    assert close(y1, y2, 1e-11) and close(d1, d2, 1e-11)
    y3, d3 = oracle.causal_mhla_stream(q, k, v, np.ones((2, 4, 4)), 24, 1e-6)
    ref, dref = oracle.causal_recurrent(q, k, v, 1e-6)
    assert close(y3, ref, 1e-11) and close(d3, dref, 1e-11)


# ------------------------------------------- feature maps, normaliser, decay
def test_other_feature_maps_closed_forms():
    assert oracle.phi_relu(-1.0) == 0.0 and oracle.phi_relu(0.0) == 0.0 and oracle.phi_relu(2.0) == 2.0
    assert oracle.phi_exp(0.0) == 1.0
    assert math.isclose(oracle.phi_exp(math.log(2.0)), 2.0, rel_tol=1e-15)


@pytest.mark.parametrize("feature", ["elu1", "relu", "exp"])
@pytest.mark.parametrize("normalise", [True, False])
def test_feature_block_form_equals_token_expansion(feature, normalise):
    q = normal(31, 1, (2, 2, 48, 6), 0.6)
    k = normal(31, 2, (2, 2, 48, 6), 0.6)
    v = normal(31, 3, (2, 2, 48, 6))
    u = uniform(31, 4, (2, 4, 4)) + 0.05
    mix = u / u.sum(axis=-1, keepdims=True)
    y1, d1 = oracle.mhla_block_form_feature(q, k, v, mix, 12, feature, 1e-6, normalise)
    y2, d2 = oracle.mhla_token_expansion_feature(q, k, v, mix, 12, feature, 1e-6, normalise)
    assert close(y1, y2, 1e-11) and close(d1, d2, 1e-11)
    if feature == "elu1":  # the default map is the block form's own
        ref, dref = oracle.mhla_block_form(q, k, v, mix, 12, 1e-6)
        assert close(d1, dref, 1e-11)
        assert close(y1, ref if normalise else ref * dref[..., None], 1e-11)


def test_relu_features_of_nonpositive_queries_give_zero():
    q = -np.abs(normal(32, 1, (1, 2, 16, 4)))
    k = normal(32, 2, (1, 2, 16, 4))
    v = normal(32, 3, (1, 2, 16, 4))
    mix = np.ones((2, 2, 2))
    for fn in (oracle.mhla_block_form_feature, oracle.mhla_token_expansion_feature):
        y, den = fn(q, k, v, mix, 8, "relu", 1e-6)
        assert np.all(y == 0.0) and np.all(den == 1e-6)


def test_exp_feature_by_hand():
    # d = 1, one block: phi(q) = 1, phi(k) = (1, 2), v = (1, 3):
    # Y = (1*1*1 + 1*2*3) / (1 + 2 + eps) for both queries, which share phi(q) = 1
    q = as4([[0.0], [0.0]])
    k = as4([[0.0], [math.log(2.0)]])
    v = as4([[1.0], [3.0]])
    for fn in (oracle.mhla_block_form_feature, oracle.mhla_token_expansion_feature):
        y, den = fn(q, k, v, np.ones((1, 1, 1)), 2, "exp", 0.0)
        assert close(y[0, 0, :, 0], [7.0 / 3.0, 7.0 / 3.0], 1e-14) and close(den[0, 0], [3.0, 3.0], 1e-14)


@pytest.mark.parametrize("feature", ["elu1", "relu", "exp"])
@pytest.mark.parametrize("gamma", [1.0, 0.9, 0.5])
def test_causal_variant_recurrence_equals_bruteforce(causal_small, feature, gamma):
    q, k, v = causal_small
    for normalise in (True, False):
        y1, d1 = oracle.causal_variant_recurrent(q, k, v, feature, gamma, 1e-6, normalise)
        y2, d2 = oracle.causal_variant_bruteforce(q, k, v, feature, gamma, 1e-6, normalise)
        assert close(y1, y2, 1e-10) and close(d1, d2, 1e-10)


def test_causal_variants_reduce_to_the_pinned_forms(causal_small):
    q, k, v = causal_small
    y, d = oracle.causal_variant_bruteforce(q, k, v)
    ref, dref = oracle.causal_bruteforce(q, k, v, 1e-6)
    assert close(y, ref, 1e-11) and close(d, dref, 1e-11)
    y, d = oracle.causal_variant_bruteforce(q, k, v, "elu1", 0.8)
    ref, dref = oracle.decayed_causal_bruteforce(q, k, v, 0.8, 1e-6)
    assert close(y, ref, 1e-11) and close(d, dref, 1e-11)
    # gamma = 0: every token attends to itself alone, Y_t = a_tt v_t / (a_tt + eps)
    y, d = oracle.causal_variant_recurrent(q, k, v, "elu1", 0.0)
    a = np.einsum("bhtc,bhtc->bht", oracle.phi(q), oracle.phi(k))
    assert close(y, a[..., None] * v / (a + 1e-6)[..., None], 1e-12)


# ---------------------------------------------------------------- backward (dQ, dK, dV, dM)
def test_phi_grad_closed_forms_and_differences():
    assert close(oracle.phi_grad([0.0, 1.0, -1.0, 3.5]), [1.0, 1.0, math.exp(-1.0), 1.0], 1e-15)
    x = np.linspace(-3.0, 3.0, 61) + 0.013  # away from the kink at 0
    h = 1e-6
    fd = (oracle.phi(x + h) - oracle.phi(x - h)) / (2 * h)
    assert close(oracle.phi_grad(x), fd, 1e-8)


@pytest.fixture
def bwd_small():
    """B2 H2 N6 d3, blocks of 2 (M = 3): inputs, a positive mixing (den stays away from 0) and dY."""
    shape = (2, 2, 6, 3)
    q, k, v, dy = (normal(700 + i, 1, shape, 0.8) for i in range(4))
    mix = uniform(704, 2, (2, 3, 3)) + 0.1
    return q, k, v, mix, dy


def _loss(q, k, v, mix, dy, eps):
    return float(np.sum(dy * oracle.mhla_block_form(q, k, v, mix, 2, eps)[0]))


@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_backward_equals_central_differences(bwd_small, eps):
    """Every entry of dq, dk, dv and dmixing against (L(x + h) - L(x - h)) / 2h of the forward."""
    q, k, v, mix, dy = bwd_small
    grads = oracle.mhla_block_form_backward(q, k, v, mix, 2, dy, eps)
    h = 1e-6
    for which, (x, g) in enumerate(zip((q, k, v, mix), grads)):
        assert g.shape == x.shape
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            args = [q, k, v, mix]
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[which] = xp
            lp = _loss(*args, dy, eps)
            args[which] = xm
            fd[idx] = (lp - _loss(*args, dy, eps)) / (2 * h)
        assert close(g, fd, 1e-7), ("q", "k", "v", "mixing")[which]


def test_backward_euler_identities(bwd_small):
    """Y is linear in V: <dV, V> = <dY, Y> for any eps.  With eps = 0, Y is of degree 0 in the
    mixing, in phi(q_t) of each token and in phi(K) of each (b, h) slice, so the matching inner
    products vanish (phi(x) = x + 1 and phi' = 1 on positive inputs)."""
    q, k, v, mix, dy = bwd_small
    y = oracle.mhla_block_form(q, k, v, mix, 2, 0.25)[0]
    dv = oracle.mhla_block_form_backward(q, k, v, mix, 2, dy, 0.25)[2]
    assert close(np.sum(dv * v), np.sum(dy * y), 1e-12)
    qp, kp = np.abs(q) + 0.1, np.abs(k) + 0.1
    dq, dk, _, dm = oracle.mhla_block_form_backward(qp, kp, v, mix, 2, dy, 0.0)
    assert abs(np.sum(dm * mix)) < 1e-12 * np.sum(np.abs(dm * mix))
    per_token = np.einsum("bhtc,bhtc->bht", dq, qp + 1.0)
    assert np.max(np.abs(per_token)) < 1e-12 * np.max(np.abs(dq))
    per_slice = np.einsum("bhtc,bhtc->bh", dk, kp + 1.0)
    assert np.max(np.abs(per_slice)) < 1e-12 * np.sum(np.abs(dk))
