"""Planted mistakes in the oracle must be caught by its pins.

Each test swaps one oracle function for a plausibly wrong variant (on the CPU,
through monkeypatch, so the real oracle is untouched afterwards) and checks
that at least one pin in ``test_oracle_pins`` then fails.
"""

import numpy as np
import pytest

import oracle
import oracle.mhla_oracle as om
import test_oracle_pins as pins
from workloads import WORKLOADS, mhla_host


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_relu_feature_map_is_caught(monkeypatch, golden_dir):
    monkeypatch.setattr(om, "phi", lambda x: np.maximum(np.asarray(x, dtype=np.float64), 0.0) + 1.0)
    _fails(pins.test_golden_linear_attention, golden_dir)


def test_exp_feature_map_is_caught(monkeypatch, golden_dir):
    monkeypatch.setattr(om, "phi", lambda x: np.exp(np.asarray(x, dtype=np.float64)))
    _fails(pins.test_golden_linear_attention, golden_dir)


def test_transposed_mixing_is_caught(monkeypatch, golden_dir):
    real = om._check_blocks

    def transposed(n, block_size, mixing):
        m, mix = real(n, block_size, mixing)
        return m, np.swapaxes(mix, -1, -2)

    monkeypatch.setattr(om, "_check_blocks", transposed)
    _fails(pins.test_golden_mhla_two_blocks, golden_dir)


def test_dropped_eps_is_caught(monkeypatch):
    real = om.mhla_block_form
    monkeypatch.setattr(oracle, "mhla_block_form",
                        lambda q, k, v, mix, bs, eps=1e-6: real(q, k, v, mix, bs, 0.0))
    _fails(pins.test_closed_form_constant_features)


def test_transposed_summary_is_caught(monkeypatch, golden_dir):
    real = om.global_linear_attention

    def wrong(q, k, v, eps=1e-6):
        # uses S^T instead of S: phi(Q) (V^T phi(K)) -- only equal when S is symmetric
        qf, kf = om.phi(q), om.phi(k)
        kv = np.einsum("...jc,...je->...ce", kf, np.asarray(v, dtype=np.float64))
        num = np.einsum("...tc,...ce->...te", qf, np.swapaxes(kv, -1, -2))
        den = np.einsum("...tc,...c->...t", qf, kf.sum(axis=-2)) + eps
        return num / den[..., None], den

    assert real is not wrong
    monkeypatch.setattr(oracle, "global_linear_attention", wrong)
    _fails(pins.test_golden_linear_attention, golden_dir)


def test_causal_mask_without_diagonal_is_caught(monkeypatch, golden_dir):
    def strict(q, k, v, eps=1e-6):
        q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
        n = q.shape[-2]
        a = np.einsum("...tc,...sc->...ts", om.phi(q), om.phi(k)) * np.tril(np.ones((n, n)), -1)
        den = a.sum(axis=-1) + eps
        return np.einsum("...ts,...se->...te", a, v) / den[..., None], den

    monkeypatch.setattr(oracle, "causal_bruteforce", strict)
    _fails(pins.test_golden_linear_attention, golden_dir)


def test_block_offset_error_is_caught(monkeypatch):
    """An off-by-one block index (b(t) shifted by one token) breaks the two-definition agreement."""
    wl = WORKLOADS["tiny"]
    x = mhla_host(wl)
    monkeypatch.setattr(om, "block_of", lambda n, bs: np.minimum((np.arange(n) + 1) // bs, n // bs - 1))
    _fails(pins.test_block_form_equals_token_expansion_tiny, (wl, x))


# ------------------------------------------------------------- newer forms
def _causal_small():
    return pins.causal_small.__wrapped__() if hasattr(pins.causal_small, "__wrapped__") else (
        pins.normal(11, 1, (2, 2, 96, 8), 0.4), pins.normal(11, 2, (2, 2, 96, 8), 0.4),
        pins.normal(11, 3, (2, 2, 96, 8)))


def test_column_major_tile_numbering_is_caught(monkeypatch):
    def column_major(gh, gw, th, tw):
        r, c = np.divmod(np.arange(gh * gw), gw)
        return (c // tw) * (gh // th) + (r // th)
    monkeypatch.setattr(oracle, "grid_block_ids", column_major)
    _fails(pins.test_grid_block_ids_by_hand)


def test_manhattan_locality_is_caught(monkeypatch):
    def manhattan(bh, bw):
        r, c = np.divmod(np.arange(bh * bw), bw)
        dist = np.abs(r[:, None] - r[None, :]) + np.abs(c[:, None] - c[None, :]) + 0.0
        far = dist.max(axis=1, keepdims=True)
        m0 = np.where(far > 0, 1.0 - dist / np.where(far > 0, far, 1.0), 1.0)
        return m0 / m0.sum(axis=1, keepdims=True)
    monkeypatch.setattr(oracle, "locality_mixing_init", manhattan)
    _fails(pins.test_locality_init_by_hand)


def test_decay_of_the_state_only_is_caught(monkeypatch):
    """Decaying S but not z (the notes write only S) must disagree with the explicit weights."""
    def s_only(s0, z0, qs, ks, vs, eps=1e-6, gamma=1.0):
        s, z = np.asarray(s0, np.float64).copy(), np.asarray(z0, np.float64).copy()
        qs, ks, vs = (np.asarray(a, np.float64) for a in (qs, ks, vs))
        outs, dens = np.empty_like(vs), np.empty(vs.shape[:-1])
        for t in range(qs.shape[0]):
            qt, kt = om.phi(qs[t]), om.phi(ks[t])
            s = gamma * s + kt[..., :, None] * vs[t][..., None, :]
            z = z + kt
            dn = np.einsum("...c,...c->...", qt, z) + eps
            outs[t] = np.einsum("...c,...ce->...e", qt, s) / dn[..., None]
            dens[t] = dn
        return outs, dens, s, z
    monkeypatch.setattr(oracle, "decode_steps", s_only)
    _fails(pins.test_decode_with_decay_equals_decayed_bruteforce, _causal_small())


def test_stream_without_self_weight_is_caught(monkeypatch):
    """The running summary entering the output with weight 1 instead of m_ii."""
    real = om.causal_mhla_stream

    def no_mii(q, k, v, mixing, block_size, eps=1e-6):
        mix = np.array(mixing, dtype=np.float64)
        m = mix.shape[-1]
        mix[:, np.arange(m), np.arange(m)] = 1.0
        return real(q, k, v, mix, block_size, eps)
    monkeypatch.setattr(oracle, "causal_mhla_stream", no_mii)
    _fails(pins.test_causal_mhla_stream_equals_bruteforce, _causal_small())


def test_swapped_feature_maps_are_caught(monkeypatch):
    monkeypatch.setitem(om.FEATURE_MAPS, "relu", om.phi_exp)
    _fails(pins.test_relu_features_of_nonpositive_queries_give_zero)


def test_undecayed_normaliser_in_the_variant_recurrence_is_caught(monkeypatch):
    def z_undecayed(q, k, v, feature="elu1", gamma=1.0, eps=1e-6, normalise=True):
        f = om.FEATURE_MAPS[feature]
        q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
        *lead, n, d = q.shape
        s, z = np.zeros((*lead, d, d)), np.zeros((*lead, d))
        y, den = np.empty_like(v), np.empty((*lead, n))
        for t in range(n):
            qt, kt = f(q[..., t, :]), f(k[..., t, :])
            s = gamma * s + kt[..., :, None] * v[..., t, None, :]
            z = z + kt
            dn = np.einsum("...c,...c->...", qt, z) + eps
            num = np.einsum("...c,...ce->...e", qt, s)
            y[..., t, :] = num / dn[..., None] if normalise else num
            den[..., t] = dn
        return y, den
    monkeypatch.setattr(oracle, "causal_variant_recurrent", z_undecayed)
    _fails(pins.test_causal_variant_recurrence_equals_bruteforce, _causal_small(), "elu1", 0.9)


# ------------------------------------------------------------ backward
bwd_small = pins.bwd_small  # the pins' fixture


def _mutated_backward(old, new):
    """The oracle's backward with one expression replaced (the text must occur exactly once)."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(om.mhla_block_form_backward))
    assert src.count(old) == 1, old
    ns = dict(vars(om))
    exec(compile(src.replace(old, new), "<mutated backward>", "exec"), ns)
    return ns["mhla_block_form_backward"]


BACKWARD_MUTATIONS = {
    # the denominator's path dropped from dphi(q)
    "no_dden_in_dq": ("+ dden[..., None] * z_mix[:, :, :, None, :]", ""),
    # dden without its minus sign
    "dden_sign": ("dden = -np.einsum", "dden = np.einsum"),
    # the mixing not transposed on the way back (m_bi instead of m_ib)
    "untransposed_mixing": ('np.einsum("hib,zhice->zhbce", mix, ds_mix)', 'np.einsum("hbi,zhice->zhbce", mix, ds_mix)'),
    # dV from dS instead of dS^T
    "dv_untransposed": ('np.einsum("bhmce,bhmjc->bhmje", ds, kf)', 'np.einsum("bhmec,bhmjc->bhmje", ds, kf)'),
    # z's gradient left out of dphi(k)
    "no_dz_in_dk": ("+ dz[:, :, :, None, :]", ""),
    # dM of the first sample only instead of the sum over the batch
    "dm_one_sample": ('np.einsum("zhice,zhbce->hib", ds_mix, s)', 'np.einsum("hice,hbce->hib", ds_mix[0], s[0])'),
}


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTATIONS))
def test_backward_mutation_is_caught(monkeypatch, bwd_small, name):
    monkeypatch.setattr(oracle, "mhla_block_form_backward", _mutated_backward(*BACKWARD_MUTATIONS[name]))
    _fails(pins.test_backward_equals_central_differences, bwd_small, 1e-6)


def test_backward_with_phi_prime_one_is_caught(monkeypatch, bwd_small):
    monkeypatch.setattr(om, "phi_grad", lambda x: np.ones_like(np.asarray(x, dtype=np.float64)))
    _fails(pins.test_backward_equals_central_differences, bwd_small, 1e-6)
