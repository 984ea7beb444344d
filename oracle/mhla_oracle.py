"""Plain float64 definitions of every step on the MHLA forward path.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path imports this module.

Conventions
-----------
* ``q, k, v``: arrays ``[B, H, N, d]`` (any float dtype; widened to float64).
* ``mixing``: ``[H, M, M]``; row ``i`` is the query block, column ``b`` the
  KV block (MHLA paper §4.1 "multi-head mixing" and §4.2, where entry (i, j)
  is the affinity of query block i to the summary of block j).
* blocks are contiguous token ranges of ``block_size`` tokens,
  ``M = N / block_size`` (MHLA paper §4.1 splits the sequence into M
  non-overlapping blocks; the contiguous 1-D reading is the one this library
  implements).
* ``eps`` is added to the denominator after mixing, as the Linear Attention
  notes do in both of their code examples (§四 and §五).

Every function is a direct transcription of the formula it cites, written
for a reader to check by eye; there is no blocking, fusion or reordering
beyond what that formula states.
"""

from __future__ import annotations

import numpy as np

# What pins each function to something other than itself
# (tests/test_oracle_pins.py holds the pins).
PIN_STATUS = {
    "phi": "closed-form values at 0, +1, -1, continuity, positivity",
    "mhla_block_form": "token-level expansion (brute N x N), closed form at Q=K=0, "
                       "identity / all-ones / row-scaled mixing, token permutation",
    "mhla_token_expansion": "closed form at Q=K=0, hand-derived golden fixture, rank bounds",
    "mhla_attention_matrix": "rank <= d for all-ones mixing, generic rank = sum_b min(n_b, d)",
    "global_linear_attention": "equals MHLA with M=1 and with all-ones mixing; golden fixture",
    "causal_recurrent": "hand-derived golden fixture; equals masked brute force",
    "causal_chunked": "equals recurrence and brute force for C in {1, 16, 64, N} and ragged C",
    "causal_bruteforce": "hand-derived golden fixture; last row equals non-causal global LA",
    "causal_mhla_chunked": "equals its masked brute force; all-ones mixing equals causal LA",
    "causal_mhla_bruteforce": "all-ones mixing equals causal_bruteforce; golden fixture",
    "decode_steps": "equals rows of the causal forward on prefix+steps; final state = sum phi(k) v^T; "
                    "with decay: equals decayed_causal_bruteforce",
    "decayed_causal_bruteforce": "gamma = 1 equals causal_bruteforce; gamma = 0 keeps only the token itself "
                                 "(out = v); hand-computed two-token value",
    "mhla_block_form_unnormalized": "equals the brute-force sum without the division; Y * den of the block form",
    "grid_block_ids": "hand-listed ids of a 4 x 4 grid in 2 x 2 tiles",
    "mhla_block_form_ids": "equals its token expansion; contiguous ids equal mhla_block_form; "
                           "equals the block form of the tile-permuted tokens",
    "mhla_token_expansion_ids": "equals mhla_token_expansion for contiguous ids",
    "locality_mixing_init": "hand-computed 1 x 3 and 2 x 2 grids; rows sum to 1, diagonal largest",
    "causal_mhla_stream": "equals causal_mhla_bruteforce; all-ones mixing equals causal linear attention",
    "phi_relu": "closed-form values at -1, 0, 2",
    "phi_exp": "closed-form values at 0, ln 2",
    "mhla_block_form_feature": "equals its token expansion for each feature map and with / without the "
                               "normaliser; ReLU with Q <= 0 gives Y = 0, den = eps; hand-derived d = 1 "
                               "exp example; elu1 equals mhla_block_form",
    "mhla_token_expansion_feature": "hand-derived d = 1 exp example; ReLU with Q <= 0 gives Y = 0",
    "causal_variant_recurrent": "equals its brute force for every feature and decay; gamma = 1, elu1 equals "
                                "causal_bruteforce; gamma = 0 keeps only the token itself",
    "causal_variant_bruteforce": "gamma = 1, elu1 equals causal_bruteforce; decayed elu1 equals "
                                 "decayed_causal_bruteforce; gamma = 0 closed form",
    "rala_forward": "brute form; closed forms at Q=0 and K=0; softmax weights sum to 1",
    "rala_bruteforce": "closed forms at Q=0 and K=0; hand-derived golden fixture",
    "numerical_rank": "diagonal matrices of known rank",
    "phi_grad": "closed-form values at 0, +1, -1; central differences of phi",
    "mhla_block_form_backward": "central differences of mhla_block_form for every entry of q, k, v and the "
                                "mixing; Euler identities: <dV, V> = <dY, Y> (Y linear in V), and with "
                                "eps = 0 <dM, M> = 0 and <dphi(q_t), phi(q_t)> = 0 per token, "
                                "sum_j <dphi(k_j), phi(k_j)> = 0 per slice (Y of degree 0 in each)",
}


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def phi(x):
    """Feature map phi(x) = ELU(x) + 1, i.e. x + 1 for x > 0 and exp(x) otherwise.

    Linear Attention notes §二 (first listed kernel choice, "ELU(x)+1") and
    its code examples; RALA notes "核函数选择" (kernel choice Elu(.)+1).  ELU
    with alpha = 1, so both branches meet at phi(0) = 1.
    """
    x = _f64(x)
    return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def block_of(n_tokens: int, block_size: int) -> np.ndarray:
    """b(t): index of the contiguous block holding token t (MHLA paper §4.2)."""
    return np.arange(n_tokens) // block_size


def _check_blocks(n, block_size, mixing):
    if block_size <= 0 or n % block_size != 0:
        raise ValueError("N must be a positive multiple of block_size")
    m = n // block_size
    mixing = _f64(mixing)
    if mixing.shape[-2:] != (m, m):
        raise ValueError(f"mixing must be [H, {m}, {m}]")
    return m, mixing


def mhla_block_form(q, k, v, mixing, block_size, eps=1e-6):
    """MHLA forward in its block form.  Returns ``(Y, den)``.

    MHLA paper §4.1:
      * local KV summary and normaliser of block b:
        S_b = sum_{j in b} phi(K_j) V_j^T  (d x d),  z_b = sum_{j in b} phi(K_j);
      * multi-head mixing for query block i:
        S~_i = sum_b m_{i,b} S_b,  z~_i = sum_b m_{i,b} z_b;
      * output for a query q in block i:
        o = phi(q)^T S~_i / (phi(q)^T z~_i)   (+ eps, Linear Attention notes §五).

    ``den`` is phi(q)^T z~_i + eps for every token, shape [B, H, N].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    m, mix = _check_blocks(n, block_size, mixing)
    kb = phi(k).reshape(bsz, nh, m, block_size, d)
    vb = v.reshape(bsz, nh, m, block_size, d)
    # S_b[c, e] = sum_j phi(k_j)_c v_j,e ; z_b[c] = sum_j phi(k_j)_c
    s = np.einsum("bhmjc,bhmje->bhmce", kb, vb)
    z = kb.sum(axis=3)
    # S~_i = sum_b m_{i,b} S_b ; z~_i = sum_b m_{i,b} z_b  (one matrix per head)
    s_mix = np.einsum("hib,zhbce->zhice", mix, s)
    z_mix = np.einsum("hib,zhbc->zhic", mix, z)
    qb = phi(q).reshape(bsz, nh, m, block_size, d)
    num = np.einsum("bhitc,bhice->bhite", qb, s_mix)
    den = np.einsum("bhitc,bhic->bhit", qb, z_mix) + eps
    y = num / den[..., None]
    return y.reshape(bsz, nh, n, d), den.reshape(bsz, nh, n)


def mhla_attention_matrix(q1, k1, mixing1, block_size):
    """Explicit MHLA attention matrix of one head, [N, N].

    MHLA paper §4.2 (token-level effect, eq. 5) and §4.3: the score of query
    t on key s is m_{b(t), b(s)} * phi(q_t)^T phi(k_s).  ``q1, k1``: [N, d];
    ``mixing1``: [M, M].
    """
    q1, k1 = _f64(q1), _f64(k1)
    n = q1.shape[0]
    _, mix = _check_blocks(n, block_size, mixing1)
    bt = block_of(n, block_size)
    kernel = phi(q1) @ phi(k1).T          # phi(q_t)^T phi(k_s)
    return mix[bt[:, None], bt[None, :]] * kernel


def mhla_token_expansion(q, k, v, mixing, block_size, eps=1e-6):
    """MHLA forward written token by token (brute force, O(N^2)).  Returns ``(Y, den)``.

    MHLA paper §4.2 eq. 5 and App. B: phi(q)^T S~_i = sum_t m_{i,b(t)}
    (phi(q)^T phi(K_t)) V_t^T, and the normaliser is the same sum without
    V_t.  For every (batch, head) this builds the N x N score matrix A and
    returns Y_t = sum_s A_ts v_s / (sum_s A_ts + eps).  Small inputs only.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    _, mix = _check_blocks(n, block_size, mixing)
    y = np.empty_like(v)
    den = np.empty((bsz, nh, n))
    for b in range(bsz):
        for h in range(nh):
            a = mhla_attention_matrix(q[b, h], k[b, h], mix[h], block_size)
            den[b, h] = a.sum(axis=1) + eps
            y[b, h] = (a @ v[b, h]) / den[b, h][:, None]
    return y, den


def global_linear_attention(q, k, v, eps=1e-6):
    """Non-causal global linear attention.  Returns ``(Y, den)``.

    Linear Attention notes §三 and §五 (parallel form): KV = phi(K)^T V
    (d x d), z = sum_j phi(K_j), Y = phi(Q) KV / (phi(Q) z + eps).  MHLA paper
    §3.1 gives the same G and z as the single global summary.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    qf, kf = phi(q), phi(k)
    kv = np.einsum("...jc,...je->...ce", kf, v)
    z = kf.sum(axis=-2)
    num = np.einsum("...tc,...ce->...te", qf, kv)
    den = np.einsum("...tc,...c->...t", qf, z) + eps
    return num / den[..., None], den


def causal_recurrent(q, k, v, eps=1e-6):
    """Causal linear attention by its recurrence.  Returns ``(Y, den)``.

    Linear Attention notes §四: S_t = S_{t-1} + phi(k_t) v_t^T,
    z_t = z_{t-1} + phi(k_t), out_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps);
    the state is updated before it is read, so token t sees itself.
    Works on any leading batch dimensions; loops over tokens in Python.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    *lead, n, d = q.shape
    s = np.zeros((*lead, d, d))
    z = np.zeros((*lead, d))
    y = np.empty_like(v)
    den = np.empty((*lead, n))
    for t in range(n):
        qt, kt, vt = phi(q[..., t, :]), phi(k[..., t, :]), v[..., t, :]
        s = s + kt[..., :, None] * vt[..., None, :]
        z = z + kt
        num = np.einsum("...c,...ce->...e", qt, s)
        dn = np.einsum("...c,...c->...", qt, z) + eps
        y[..., t, :] = num / dn[..., None]
        den[..., t] = dn
    return y, den


def causal_bruteforce(q, k, v, eps=1e-6):
    """Causal linear attention from the explicit masked N x N matrix.  Returns ``(Y, den)``.

    Linear Attention notes §三 (out_i = sum_j phi(q_i)^T phi(k_j) v_j over the
    normaliser) with the causal mask of the Attention tutorial ("Mask"): only
    the strictly upper triangle (future keys) is removed, the diagonal stays.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[-2]
    a = np.einsum("...tc,...sc->...ts", phi(q), phi(k))
    a = a * np.tril(np.ones((n, n)))
    den = a.sum(axis=-1) + eps
    return np.einsum("...ts,...se->...te", a, v) / den[..., None], den


def causal_chunked(q, k, v, chunk, eps=1e-6):
    """Chunkwise-parallel causal linear attention.  Returns ``(Y, den)``.

    MHLA paper App. C: for chunk i, the output is the inter-chunk term
    phi(Q_i) S^global_{i-1} plus the intra-chunk term (phi(Q_i) phi(K_i)^T) V_i,
    then S^global_i = S^global_{i-1} + S_i.  The intra-chunk scores keep the
    lower triangle including the diagonal (Attention tutorial "Mask"), and the
    normaliser is built the same way with eps (Linear Attention notes §四).
    The last chunk may be shorter than ``chunk``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    *lead, n, d = q.shape
    if chunk <= 0:
        raise ValueError("chunk must be positive")
    p = np.zeros((*lead, d, d))     # S^global of all previous chunks
    zeta = np.zeros((*lead, d))     # sum of phi(K) over all previous chunks
    y = np.empty_like(v)
    den = np.empty((*lead, n))
    for c0 in range(0, n, chunk):
        c1 = min(c0 + chunk, n)
        qc, kc, vc = phi(q[..., c0:c1, :]), phi(k[..., c0:c1, :]), v[..., c0:c1, :]
        length = c1 - c0
        intra = np.einsum("...tc,...sc->...ts", qc, kc) * np.tril(np.ones((length, length)))
        num = np.einsum("...tc,...ce->...te", qc, p) + np.einsum("...ts,...se->...te", intra, vc)
        dn = np.einsum("...tc,...c->...t", qc, zeta) + intra.sum(axis=-1) + eps
        y[..., c0:c1, :] = num / dn[..., None]
        den[..., c0:c1] = dn
        p = p + np.einsum("...sc,...se->...ce", kc, vc)
        zeta = zeta + kc.sum(axis=-2)
    return y, den


def causal_mhla_chunked(q, k, v, mixing, block_size, eps=1e-6):
    """Causal MHLA with a lower-triangular mixing matrix, chunk = block.  Returns ``(Y, den)``.

    MHLA paper §4.2 ("chunkwise-parallel form": mixed prefix summary
    S~_i = sum_{b<=i} m_{i,b} S_b) and App. C.  App. C's printed formula is
    garbled; the reading implemented is
      H_i = phi(Q_i) (sum_{b<i} m_{i,b} S_b) + m_{i,i} tril(phi(Q_i) phi(K_i)^T) V_i
    with the normaliser built the same way plus eps.  Entries of ``mixing``
    above the diagonal are ignored (the paper masks them).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    m, mix = _check_blocks(n, block_size, mixing)
    qb = phi(q).reshape(bsz, nh, m, block_size, d)
    kb = phi(k).reshape(bsz, nh, m, block_size, d)
    vb = v.reshape(bsz, nh, m, block_size, d)
    s = np.einsum("bhmjc,bhmje->bhmce", kb, vb)
    z = kb.sum(axis=3)
    tri = np.tril(np.ones((block_size, block_size)))
    y = np.empty((bsz, nh, m, block_size, d))
    den = np.empty((bsz, nh, m, block_size))
    for i in range(m):
        w_prev = mix[:, i, :i]                                   # [H, i]
        s_prev = np.einsum("hb,zhbce->zhce", w_prev, s[:, :, :i])
        z_prev = np.einsum("hb,zhbc->zhc", w_prev, z[:, :, :i])
        intra = np.einsum("zhtc,zhsc->zhts", qb[:, :, i], kb[:, :, i]) * tri
        intra = intra * mix[:, i, i][None, :, None, None]
        num = np.einsum("zhtc,zhce->zhte", qb[:, :, i], s_prev) + \
            np.einsum("zhts,zhse->zhte", intra, vb[:, :, i])
        dn = np.einsum("zhtc,zhc->zht", qb[:, :, i], z_prev) + intra.sum(axis=-1) + eps
        y[:, :, i] = num / dn[..., None]
        den[:, :, i] = dn
    return y.reshape(bsz, nh, n, d), den.reshape(bsz, nh, n)


def causal_mhla_bruteforce(q, k, v, mixing, block_size, eps=1e-6):
    """Causal MHLA from the explicit masked, mixed N x N score matrix.  Returns ``(Y, den)``.

    Score of query t on key s: m_{b(t), b(s)} phi(q_t)^T phi(k_s) for s <= t
    (MHLA paper §4.2 eq. 5 restricted by the causal mask of the Attention
    tutorial), zero otherwise.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    _, mix = _check_blocks(n, block_size, mixing)
    tri = np.tril(np.ones((n, n)))
    y = np.empty_like(v)
    den = np.empty((bsz, nh, n))
    for b in range(bsz):
        for h in range(nh):
            a = mhla_attention_matrix(q[b, h], k[b, h], mix[h], block_size) * tri
            den[b, h] = a.sum(axis=1) + eps
            y[b, h] = (a @ v[b, h]) / den[b, h][:, None]
    return y, den


def decode_steps(s0, z0, qs, ks, vs, eps=1e-6, gamma=1.0):
    """Recurrent decode: T single-token steps from state (S, z).

    Linear Attention notes §四 (and §八: the state is a fixed-size d x d
    "KV cache"): per step S <- S + phi(k) v^T, z <- z + phi(k), then
    out = phi(q)^T S / (phi(q)^T z + eps).  With ``gamma`` the RetNet decay of
    the notes' §七, S <- gamma S + phi(k) v^T; the normaliser z decays the same
    way (the notes write only S; the reading keeps out a weighted mean).
    ``s0``: [..., d, d] with S[c, e] = sum phi(k)_c v_e; ``z0``: [..., d];
    ``qs, ks, vs``: [T, ..., d].  Returns ``(outs [T, ..., d], dens [T, ...], S_T, z_T)``.
    """
    s, z = _f64(s0).copy(), _f64(z0).copy()
    qs, ks, vs = _f64(qs), _f64(ks), _f64(vs)
    outs = np.empty_like(vs)
    dens = np.empty(vs.shape[:-1])
    for t in range(qs.shape[0]):
        qt, kt = phi(qs[t]), phi(ks[t])
        s = gamma * s + kt[..., :, None] * vs[t][..., None, :]
        z = gamma * z + kt
        dn = np.einsum("...c,...c->...", qt, z) + eps
        outs[t] = np.einsum("...c,...ce->...e", qt, s) / dn[..., None]
        dens[t] = dn
    return outs, dens, s, z


def decayed_causal_bruteforce(q, k, v, gamma, eps=1e-6, s0=None, z0=None):
    """Causal linear attention with RetNet decay from its explicit weights.  Returns ``(Y, den)``.

    Linear Attention notes §七: unrolling S_t = gamma S_{t-1} + phi(k_t) v_t^T
    from an initial state S_{-1} = s0 gives S_t = gamma^(t+1) s0 +
    sum_{s<=t} gamma^(t-s) phi(k_s) v_s^T (z likewise); out_t = phi(q_t)^T S_t
    / (phi(q_t)^T z_t + eps).  The score of query t on key s is
    gamma^(t-s) phi(q_t)^T phi(k_s) for s <= t.  ``q, k, v``: [..., N, d];
    ``s0, z0`` default to zero.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    *lead, n, d = q.shape
    t = np.arange(n)
    w = np.where(t[:, None] >= t[None, :], float(gamma) ** np.maximum(t[:, None] - t[None, :], 0), 0.0)
    qf = phi(q)
    a = np.einsum("...tc,...sc->...ts", qf, phi(k)) * w
    num = np.einsum("...ts,...se->...te", a, v)
    dn = a.sum(axis=-1) + eps
    if s0 is not None:
        g = float(gamma) ** (t + 1)
        num = num + g[:, None] * np.einsum("...tc,...ce->...te", qf, _f64(s0))
        dn = dn + g * np.einsum("...tc,...c->...t", qf, _f64(z0))
    return num / dn[..., None], dn


def phi_relu(x):
    """Feature map phi(x) = ReLU(x) = max(x, 0): Linear Attention notes §二 (third listed choice)."""
    return np.maximum(_f64(x), 0.0)


def phi_exp(x):
    """Feature map phi(x) = exp(x): Linear Attention notes §二 (second listed choice)."""
    return np.exp(_f64(x))


# Linear Attention notes §二's kernel choices by name.
FEATURE_MAPS = {"elu1": phi, "relu": phi_relu, "exp": phi_exp}


def mhla_block_form_feature(q, k, v, mixing, block_size, feature="elu1", eps=1e-6, normalise=True):
    """MHLA block form with the feature map of the Linear Attention notes §二 named by
    ``feature``, and with the normaliser left out when ``normalise`` is false (MHLA paper §4.1:
    it may be omitted; then Y is the numerator alone).  Returns ``(Y, den)``; ``den`` is the
    denominator phi(q)^T z~ + eps either way.

    S_b = sum_{t in b} phi(k_t) v_t^T, z_b = sum_{t in b} phi(k_t); S~_i = sum_b m_ib S_b;
    Y_t = phi(q_t)^T S~_{b(t)} [/ (phi(q_t)^T z~_{b(t)} + eps)].
    """
    f = FEATURE_MAPS[feature]
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    m, mix = _check_blocks(n, block_size, mixing)
    kb = f(k).reshape(bsz, nh, m, block_size, d)
    vb = v.reshape(bsz, nh, m, block_size, d)
    s_b = np.einsum("bhmjc,bhmje->bhmce", kb, vb)
    z_b = kb.sum(axis=3)
    s_mix = np.einsum("hib,zhbce->zhice", mix, s_b)
    z_mix = np.einsum("hib,zhbc->zhic", mix, z_b)
    qb = f(q).reshape(bsz, nh, m, block_size, d)
    num = np.einsum("bhitc,bhice->bhite", qb, s_mix).reshape(bsz, nh, n, d)
    den = np.einsum("bhitc,bhic->bhit", qb, z_mix).reshape(bsz, nh, n) + eps
    return (num / den[..., None] if normalise else num), den


def mhla_token_expansion_feature(q, k, v, mixing, block_size, feature="elu1", eps=1e-6, normalise=True):
    """Brute force of :func:`mhla_block_form_feature`: scores A_ts = m_{b(t),b(s)}
    phi(q_t)^T phi(k_s) (MHLA paper §4.2 eq. 5 with the notes' §二 feature map),
    Y_t = sum_s A_ts v_s [/ (sum_s A_ts + eps)].  Returns ``(Y, den)``."""
    f = FEATURE_MAPS[feature]
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[-2]
    _, mix = _check_blocks(n, block_size, mixing)
    b = block_of(n, block_size)
    a = np.einsum("zhtc,zhsc->zhts", f(q), f(k)) * mix[:, b[:, None], b[None, :]][None]
    den = a.sum(axis=-1) + eps
    num = np.einsum("zhts,zhse->zhte", a, v)
    return (num / den[..., None] if normalise else num), den


def causal_variant_recurrent(q, k, v, feature="elu1", gamma=1.0, eps=1e-6, normalise=True):
    """Causal linear attention by its recurrence with the notes' variants.  Returns ``(Y, den)``.

    Linear Attention notes §四 recurrence, §七 RetNet decay (S_t = gamma S_{t-1} + phi(k_t)
    v_t^T; z decays the same way) and §二 feature map; MHLA paper §4.1: without the
    normaliser Y_t = phi(q_t)^T S_t.  ``q, k, v``: [..., N, d].
    """
    f = FEATURE_MAPS[feature]
    q, k, v = _f64(q), _f64(k), _f64(v)
    *lead, n, d = q.shape
    s = np.zeros((*lead, d, d))
    z = np.zeros((*lead, d))
    y = np.empty_like(v)
    den = np.empty((*lead, n))
    for t in range(n):
        qt, kt = f(q[..., t, :]), f(k[..., t, :])
        s = gamma * s + kt[..., :, None] * v[..., t, None, :]
        z = gamma * z + kt
        dn = np.einsum("...c,...c->...", qt, z) + eps
        num = np.einsum("...c,...ce->...e", qt, s)
        y[..., t, :] = num / dn[..., None] if normalise else num
        den[..., t] = dn
    return y, den


def causal_variant_bruteforce(q, k, v, feature="elu1", gamma=1.0, eps=1e-6, normalise=True):
    """Causal linear attention with the notes' variants from the explicit weights
    gamma^(t-s) phi(q_t)^T phi(k_s), s <= t (Linear Attention notes §七 unrolled, §二 feature
    map; MHLA paper §4.1 for the optional normaliser).  Returns ``(Y, den)``."""
    f = FEATURE_MAPS[feature]
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[-2]
    t = np.arange(n)
    w = np.where(t[:, None] >= t[None, :], float(gamma) ** np.maximum(t[:, None] - t[None, :], 0), 0.0)
    a = np.einsum("...tc,...sc->...ts", f(q), f(k)) * w
    num = np.einsum("...ts,...se->...te", a, v)
    dn = a.sum(axis=-1) + eps
    return (num / dn[..., None] if normalise else num), dn


def _rala_weights(q1, k1):
    """Softmax weights alpha_j of one (batch, head): RALA notes, KV buffer rank augmentation.

    Q_g is the mean of the raw queries over all tokens; alpha = softmax over
    tokens j of Q_g^T phi(K_j).  The maximum is subtracted before exp, which
    leaves alpha unchanged in exact arithmetic.
    """
    q_g = q1.mean(axis=0)
    logits = phi(k1) @ q_g
    e = np.exp(logits - logits.max())
    return e / e.sum()


def rala_forward(q, k, v, x, w):
    """Rank-augmented linear attention (RALA) forward.  Returns Y [B, H, N, d].

    RALA notes, "关键设计" (key designs):
      1. KV buffer rank augmentation: Q_g = mean_i Q_i,
         alpha_j = softmax_j(Q_g^T phi(K_j)), B = sum_j alpha_j phi(K_j)^T V_j;
      2. output rank augmentation: Y_i = phi_X(X_i) * (phi(Q_i) B) (Hadamard
         product), with phi_X the linear map X W; ``x``: [B, N, Cx] shared by
         all heads of a sample, ``w``: [Cx, d] shared by all heads.
    No normaliser and no eps appear in the notes' output formula.
    """
    q, k, v, x, w = _f64(q), _f64(k), _f64(v), _f64(x), _f64(w)
    bsz, nh, n, d = q.shape
    y = np.empty_like(v)
    for b in range(bsz):
        gate = x[b] @ w                                   # [N, d]
        for h in range(nh):
            alpha = _rala_weights(q[b, h], k[b, h])
            buf = np.einsum("j,jc,je->ce", alpha, phi(k[b, h]), v[b, h])
            y[b, h] = gate * (phi(q[b, h]) @ buf)
    return y


def rala_bruteforce(q, k, v, x, w):
    """RALA written token by token: Y_t = (X W)_t * sum_s alpha_s (phi(q_t)^T phi(k_s)) v_s.

    Same definitions as ``rala_forward`` (RALA notes, key designs 1 and 2)
    with the d x d buffer B expanded into its token sum.  Small inputs only.
    """
    q, k, v, x, w = _f64(q), _f64(k), _f64(v), _f64(x), _f64(w)
    bsz, nh, n, d = q.shape
    y = np.empty_like(v)
    for b in range(bsz):
        gate = x[b] @ w
        for h in range(nh):
            alpha = _rala_weights(q[b, h], k[b, h])
            scores = (phi(q[b, h]) @ phi(k[b, h]).T) * alpha[None, :]
            y[b, h] = gate * (scores @ v[b, h])
    return y


def mhla_block_form_unnormalized(q, k, v, mixing, block_size):
    """MHLA forward without the normaliser: Y_t = phi(q_t)^T S~_{b(t)}.

    MHLA paper §4.1 ("the normalisation term can be omitted" for long
    sequences in language and video models): the block form's numerator.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    m, mix = _check_blocks(n, block_size, mixing)
    kb = phi(k).reshape(bsz, nh, m, block_size, d)
    vb = v.reshape(bsz, nh, m, block_size, d)
    s = np.einsum("bhmjc,bhmje->bhmce", kb, vb)
    s_mix = np.einsum("hib,zhbce->zhice", mix, s)
    qb = phi(q).reshape(bsz, nh, m, block_size, d)
    return np.einsum("bhitc,bhice->bhite", qb, s_mix).reshape(bsz, nh, n, d)


def grid_block_ids(grid_h, grid_w, tile_h, tile_w):
    """b(t) for tokens on a grid_h x grid_w grid in row-major order, blocks the tile_h x
    tile_w tiles, numbered row-major over the (grid_h / tile_h) x (grid_w / tile_w) tile grid.

    MHLA paper §4.1: in vision models the blocks lie on 2-D (or 3-D) grids;
    Fig. 4b shows M = 25 blocks as a 5 x 5 grid.
    """
    if grid_h % tile_h or grid_w % tile_w:
        raise ValueError("the tiles must cover the grid")
    r, c = np.divmod(np.arange(grid_h * grid_w), grid_w)
    return (r // tile_h) * (grid_w // tile_w) + (c // tile_w)


def mhla_block_form_ids(q, k, v, mixing, block_ids, eps=1e-6):
    """MHLA forward with blocks given token by token (``block_ids[t]`` = b(t)).  Returns ``(Y, den)``.

    MHLA paper §4.1 with blocks that need not be contiguous token ranges:
    S_b = sum_{t: b(t)=b} phi(K_t) V_t^T, z_b = sum_{t: b(t)=b} phi(K_t),
    S~_i = sum_b m_ib S_b, Y_t = phi(q_t)^T S~_{b(t)} / (phi(q_t)^T z~_{b(t)} + eps).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    ids = np.asarray(block_ids)
    m = int(ids.max()) + 1
    mix = _f64(mixing)
    if mix.shape[-2:] != (m, m):
        raise ValueError(f"mixing must be [H, {m}, {m}]")
    onehot = (ids[None, :] == np.arange(m)[:, None]).astype(np.float64)  # [M, N]
    kf = phi(k)
    s = np.einsum("bt,zhtc,zhte->zhbce", onehot, kf, v)
    z = np.einsum("bt,zhtc->zhbc", onehot, kf)
    s_mix = np.einsum("hib,zhbce->zhice", mix, s)
    z_mix = np.einsum("hib,zhbc->zhic", mix, z)
    qf = phi(q)
    num = np.einsum("zhtc,zhtce->zhte", qf, s_mix[:, :, ids])
    den = np.einsum("zhtc,zhtc->zht", qf, z_mix[:, :, ids]) + eps
    return num / den[..., None], den


def mhla_token_expansion_ids(q, k, v, mixing, block_ids, eps=1e-6):
    """Brute force of :func:`mhla_block_form_ids`: the N x N scores m_{b(t), b(s)}
    phi(q_t)^T phi(k_s) (MHLA paper §4.2 eq. 5), Y_t = sum_s A_ts v_s / (sum_s A_ts + eps)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    ids = np.asarray(block_ids)
    mix = _f64(mixing)
    a = np.einsum("zhtc,zhsc->zhts", phi(q), phi(k)) * mix[:, ids[:, None], ids[None, :]][None]
    den = a.sum(axis=-1) + eps
    return np.einsum("zhts,zhse->zhte", a, v) / den[..., None], den


def locality_mixing_init(blocks_h, blocks_w):
    """Locality-based initial mixing matrix for blocks on a blocks_h x blocks_w grid.  [M, M].

    MHLA paper §4.2: m^(0)_{i,j} proportional to 1 - dist(i, j) / max_k dist(i, k),
    dist the Euclidean distance between the blocks' grid positions, each row
    then normalised to sum to 1.  With a single block the row is [1].
    """
    r, c = np.divmod(np.arange(blocks_h * blocks_w), blocks_w)
    dist = np.sqrt((r[:, None] - r[None, :]) ** 2.0 + (c[:, None] - c[None, :]) ** 2.0)
    far = dist.max(axis=1, keepdims=True)
    m0 = np.where(far > 0, 1.0 - dist / np.where(far > 0, far, 1.0), 1.0)
    return m0 / m0.sum(axis=1, keepdims=True)


def causal_mhla_stream(q, k, v, mixing, block_size, eps=1e-6):
    """Causal MHLA inference, one token at a time.  Returns ``(Y, den)``.

    MHLA paper App. C ("因果推理"): the summaries of finished blocks are frozen;
    for a token of block i the running summary of block i takes the token
    (S_i <- S_i + phi(k) v^T, z_i <- z_i + phi(k)) and the output reads the
    mixture sum_{b<i} m_{i,b} S_b + m_{i,i} S_i (z likewise), then divides
    as everywhere else (the reading of :func:`causal_mhla_chunked`).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bsz, nh, n, d = q.shape
    m, mix = _check_blocks(n, block_size, mixing)
    frozen_s = np.zeros((bsz, nh, m, d, d))
    frozen_z = np.zeros((bsz, nh, m, d))
    y = np.empty_like(v)
    den = np.empty((bsz, nh, n))
    for t in range(n):
        i = t // block_size
        if t % block_size == 0:
            s_cur = np.zeros((bsz, nh, d, d))
            z_cur = np.zeros((bsz, nh, d))
        qt, kt = phi(q[:, :, t]), phi(k[:, :, t])
        s_cur = s_cur + kt[..., :, None] * v[:, :, t][..., None, :]
        z_cur = z_cur + kt
        s_mix = np.einsum("hb,zhbce->zhce", mix[:, i, :i], frozen_s[:, :, :i]) + mix[:, i, i][None, :, None, None] * s_cur
        z_mix = np.einsum("hb,zhbc->zhc", mix[:, i, :i], frozen_z[:, :, :i]) + mix[:, i, i][None, :, None] * z_cur
        dn = np.einsum("zhc,zhc->zh", qt, z_mix) + eps
        y[:, :, t] = np.einsum("zhc,zhce->zhe", qt, s_mix) / dn[..., None]
        den[:, :, t] = dn
        if t % block_size == block_size - 1:
            frozen_s[:, :, i] = s_cur
            frozen_z[:, :, i] = z_cur
    return y, den


def phi_grad(x):
    """Derivative of phi = ELU + 1: 1 for x > 0, exp(x) for x <= 0.

    Both one-sided derivatives at 0 equal 1, so phi is continuously
    differentiable (Linear Attention notes §二 feature map, ELU with alpha = 1).
    """
    x = _f64(x)
    return np.where(x > 0.0, 1.0, np.exp(np.minimum(x, 0.0)))


def mhla_block_form_backward(q, k, v, mixing, block_size, dy, eps=1e-6):
    """Gradients of the scalar sum(dy * Y), Y = mhla_block_form(q, k, v, mixing, block_size, eps)[0].
    Returns ``(dq, dk, dv, dmixing)``; ``dmixing`` is [H, M, M] and sums over the batch, since the
    mixing of head h is shared by every sample.

    MHLA paper §4.2 learns the mixing coefficients end to end but gives no backward formulas;
    these are the chain rule through the forward steps of §4.1, taken in reverse order
    (block i holds the query token t, block b the key token j):
      Y_t = num_t / den_t           -> dnum_t = dY_t / den_t,   dden_t = -(dY_t . Y_t) / den_t
      num_t = phi(q_t)^T S~_i       -> dS~_i = sum_t phi(q_t) dnum_t^T,   dphi(q_t) = S~_i dnum_t
      den_t = phi(q_t) . z~_i + eps -> dz~_i = sum_t phi(q_t) dden_t,     dphi(q_t) += dden_t z~_i
      S~_i = sum_b m_ib S_b (z too) -> dS_b = sum_i m_ib dS~_i,  dz_b = sum_i m_ib dz~_i,
                                       dm_ib = <dS~_i, S_b> + dz~_i . z_b   (summed over samples)
      S_b = sum_j phi(k_j) v_j^T    -> dphi(k_j) = dS_b v_j + dz_b,   dv_j = dS_b^T phi(k_j)
      z_b = sum_j phi(k_j)
      dq = phi'(q) dphi(q),  dk = phi'(k) dphi(k).
    """
    q, k, v, dy = _f64(q), _f64(k), _f64(v), _f64(dy)
    bsz, nh, n, d = q.shape
    m, mix = _check_blocks(n, block_size, mixing)
    # the forward's intermediate values (block summaries, mixed summaries, num, den)
    kf = phi(k).reshape(bsz, nh, m, block_size, d)
    vb = v.reshape(bsz, nh, m, block_size, d)
    s = np.einsum("bhmjc,bhmje->bhmce", kf, vb)
    z = kf.sum(axis=3)
    s_mix = np.einsum("hib,zhbce->zhice", mix, s)
    z_mix = np.einsum("hib,zhbc->zhic", mix, z)
    qf = phi(q).reshape(bsz, nh, m, block_size, d)
    num = np.einsum("bhitc,bhice->bhite", qf, s_mix)
    den = np.einsum("bhitc,bhic->bhit", qf, z_mix) + eps
    y = num / den[..., None]
    # Y = num / den
    g = dy.reshape(bsz, nh, m, block_size, d)
    dnum = g / den[..., None]
    dden = -np.einsum("bhite,bhite->bhit", g, y) / den
    # num and den
    ds_mix = np.einsum("bhitc,bhite->bhice", qf, dnum)
    dz_mix = np.einsum("bhitc,bhit->bhic", qf, dden)
    dqf = np.einsum("bhice,bhite->bhitc", s_mix, dnum) + dden[..., None] * z_mix[:, :, :, None, :]
    # mixing
    ds = np.einsum("hib,zhice->zhbce", mix, ds_mix)
    dz = np.einsum("hib,zhic->zhbc", mix, dz_mix)
    dmix = np.einsum("zhice,zhbce->hib", ds_mix, s) + np.einsum("zhic,zhbc->hib", dz_mix, z)
    # block summaries
    dkf = np.einsum("bhmce,bhmje->bhmjc", ds, vb) + dz[:, :, :, None, :]
    dv = np.einsum("bhmce,bhmjc->bhmje", ds, kf)
    dq = phi_grad(q) * dqf.reshape(bsz, nh, n, d)
    dk = phi_grad(k) * dkf.reshape(bsz, nh, n, d)
    return dq, dk, dv.reshape(bsz, nh, n, d), dmix


def numerical_rank(a, rtol=None):
    """Numerical rank: singular values above max(shape) * eps * sigma_max (default tolerance)."""
    a = _f64(a)
    sv = np.linalg.svd(a, compute_uv=False)
    if sv.size == 0 or sv[0] == 0.0:
        return 0
    tol = (max(a.shape) * np.finfo(np.float64).eps if rtol is None else rtol) * sv[0]
    return int((sv > tol).sum())
