"""The block form of the CCQ read agrees with the sequential statement.

CCQ ("Don't Read Everything: A Curvature-Conditioned Query for Linear
Attention", gist.science 2606.01294, "O Mecanismo"): q_clean_t =
(I - lambda_t Sigma_t) q_t with Sigma_t the running covariance of the keys.
The tensor-core kernel streams blocks of tokens and carries only the sums of
the statistics (M = sum k k^T, m = sum k, n) between blocks.  With M_b, m_b,
n_b the sums before a block, and for token t of the block n_t = n_b + t + 1,
s_t = (m_t . q_t) / n_t:

    M_t q_t - s_t m_t = (Q M_b)_t - s_t m_b + sum_{s<=t} (q_t . k_s - s_t) k_s,

so with G = Q K^T and A'_ts = G_ts - s_t on and below the diagonal (0 above),
O = Q M_b + A' K, q_clean_t = q_t - lambda_t / n_t (O_t - s_t m_b), and
M_{b+1} = M_b + K^T K.  This file restates that block form in plain numpy fp64
(test only) and checks it against the oracle's token-by-token statement,
with and without carried statistics and with a ragged last block.
"""
import numpy as np
import pytest

import oracle


def ccq_blocks(q, k, lam, C, M0=None, m0=None, n0=0.0):
    T, d = q.shape
    M = np.zeros((d, d)) if M0 is None else M0.copy()
    m = np.zeros(d) if m0 is None else m0.copy()
    n = float(n0)
    out = np.zeros_like(q)
    for c0 in range(0, T, C):
        Q, K, L = q[c0:c0 + C], k[c0:c0 + C], lam[c0:c0 + C]
        nb = Q.shape[0]
        G = Q @ K.T
        n_t = n + np.arange(1, nb + 1)
        s = (Q @ m + np.cumsum(np.tril(G), axis=1)[np.arange(nb), np.arange(nb)]) / n_t
        A = np.tril(G - s[:, None])
        O = Q @ M + A @ K
        out[c0:c0 + C] = Q - (L / n_t)[:, None] * (O - s[:, None] * m[None, :])
        M = M + K.T @ K
        m = m + K.sum(axis=0)
        n += nb
    return out, (M, m, n)


def _case(seed, T, d, with_stats):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d)) + 0.3
    lam = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    if not with_stats:
        return q, k, lam, None
    k0 = rng.standard_normal((40, d))
    return q, k, lam, (k0.T @ k0, k0.sum(axis=0), 40.0)


@pytest.mark.parametrize("C", [1, 16, 128])
@pytest.mark.parametrize("with_stats", [False, True])
def test_ccq_block_form_equals_sequential(C, with_stats):
    T, d = 300, 16   # a ragged last block for C = 16 and 128
    q, k, lam, st = _case(C + 7 * with_stats, T, d, with_stats)
    stats0 = None if st is None else (st[0][None, None], st[1][None, None], np.array([[st[2]]]))
    ref, (Ms, ms, ns) = oracle.ccq_query(q[None, :, None], k[None, :, None], lam[None, :, None],
                                         stats0)
    got, (M, m, n) = ccq_blocks(q, k, lam, C, *(st if st else (None, None, 0.0)))
    scale = np.abs(ref).max()
    assert np.abs(got - ref[0, :, 0]).max() <= 1e-11 * scale
    assert np.allclose(M, Ms[0, 0], rtol=1e-12, atol=1e-9)
    assert np.allclose(m, ms[0, 0], rtol=1e-12, atol=1e-10)
    assert n == ns[0, 0]


def test_a_block_form_mistake_is_caught():
    """A' taken strictly below the diagonal (dropping each token's own key)
    must not reproduce the oracle."""
    T, d, C = 200, 16, 64
    q, k, lam, _ = _case(3, T, d, False)
    ref, _ = oracle.ccq_query(q[None, :, None], k[None, :, None], lam[None, :, None])
    ref = ref[0, :, 0]
    M, m, n = np.zeros((d, d)), np.zeros(d), 0.0
    out = np.zeros_like(q)
    for c0 in range(0, T, C):
        Q, K, L = q[c0:c0 + C], k[c0:c0 + C], lam[c0:c0 + C]
        nb = Q.shape[0]
        G = Q @ K.T
        n_t = n + np.arange(1, nb + 1)
        s = (Q @ m + np.cumsum(np.tril(G), axis=1)[np.arange(nb), np.arange(nb)]) / n_t
        A = np.tril(G - s[:, None], -1)          # the mistake
        O = Q @ M + A @ K
        out[c0:c0 + C] = Q - (L / n_t)[:, None] * (O - s[:, None] * m[None, :])
        M, m, n = M + K.T @ K, m + K.sum(axis=0), n + nb
    assert np.abs(out - ref).max() > 1e-3 * np.abs(ref).max()
