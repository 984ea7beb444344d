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
