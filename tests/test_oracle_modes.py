"""Pins for the oracle's write-coefficient modes (CPU).

"given" takes beta_t = eta_t as the write strength -- Gated DeltaNet's learned
beta, which KLA replaces by the Kaczmarz coefficient beta_t = eta_t /
(||k_t||^2 + eps) (KLA summary, gist.science 2605.08587, "Contribuicoes
Principais" item 2 and "Implementacao"); alpha = None means no decay
(DeltaNet; Linear Attention Architectures, gist.science 2607.07953,
"Metodologia e Estrutura").  Each pin is a closed form, an invariant of the
update, or the reduction of one mode to the other; a mistake planted in a
copy of the oracle source fails them.
"""
import numpy as np
import pytest

import oracle


def _case(seed, T=12, dk=6, dv=5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, dk))
    k = rng.standard_normal((1, T, 1, dk)) * rng.uniform(0.3, 3.0, (1, T, 1, 1))
    v = rng.standard_normal((1, T, 1, dv))
    alpha = rng.uniform(0.3, 1.0, (1, T, 1))
    eta = rng.uniform(0.1, 1.0, (1, T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv))
    return q, k, v, alpha, eta, S0


def test_given_mode_with_the_kaczmarz_coefficient_equals_kaczmarz_mode():
    """beta computed outside the oracle (numpy) and passed as the given write
    strength reproduces the Kaczmarz mode."""
    q, k, v, alpha, eta, S0 = _case(1)
    eps = 0.3
    n2 = np.einsum("bthd,bthd->bth", k, k)
    beta = eta / (n2 + eps)
    o1, S1 = oracle.forward(q, k, v, alpha, eta, eps, S0)
    o2, S2 = oracle.forward(q, k, v, alpha, beta, eps, S0, beta_mode="given")
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S1, rtol=1e-12, atol=1e-13)


def test_given_single_write_closed_form():
    """alpha = 1, S0 = 0, one token: S = beta k v^T and o = beta (k.q) v,
    whatever ||k|| and eps are."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 1, 4)); k = 3.0 * rng.standard_normal((1, 1, 1, 4))
    v = rng.standard_normal((1, 1, 1, 3)); beta = np.full((1, 1, 1), 0.37)
    o, S = oracle.forward(q, k, v, None, beta, 0.5, None, beta_mode="given")
    kk, vv, qq = k[0, 0, 0], v[0, 0, 0], q[0, 0, 0]
    np.testing.assert_allclose(S[0, 0], 0.37 * np.outer(kk, vv), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(o[0, 0, 0], 0.37 * (kk @ qq) * vv, rtol=1e-13, atol=1e-14)


def test_given_residual_closed_form():
    """For every token, S_t^T k_t - v_t = -(1 - beta_t ||k_t||^2) e_t with
    e_t = v_t - alpha_t S_{t-1}^T k_t: the delta-rule write with a free beta."""
    q, k, v, alpha, beta, S0 = _case(3, T=15)
    Ss = [S0[0, 0]]
    S = S0
    for t in range(q.shape[1]):
        _, S = oracle.forward(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], alpha[:, t:t + 1],
                              beta[:, t:t + 1], 1e-6, S, beta_mode="given")
        Ss.append(S[0, 0])
    for t in range(q.shape[1]):
        kt, vt = k[0, t, 0], v[0, t, 0]
        e = vt - alpha[0, t, 0] * Ss[t].T @ kt
        np.testing.assert_allclose(Ss[t + 1].T @ kt - vt, -(1 - beta[0, t, 0] * (kt @ kt)) * e,
                                   rtol=1e-10, atol=1e-12)


def test_deltanet_unit_keys_beta_one_stores_exactly():
    """DeltaNet (no decay) with unit keys and beta = 1: each write makes
    S_t^T k_t = v_t exactly."""
    rng = np.random.default_rng(4)
    T, dk, dv = 9, 5, 4
    k = rng.standard_normal((1, T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((1, T, 1, dk)); v = rng.standard_normal((1, T, 1, dv))
    S = rng.standard_normal((1, 1, dk, dv))
    for t in range(T):
        _, S = oracle.forward(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], None,
                              np.ones((1, 1, 1)), 0.0, S, beta_mode="given")
        np.testing.assert_allclose(S[0, 0].T @ k[0, t, 0], v[0, t, 0], rtol=1e-12, atol=1e-13)


def test_no_decay_equals_unit_decay():
    q, k, v, alpha, eta, S0 = _case(5)
    ones = np.ones_like(alpha)
    for mode in ("kaczmarz", "given"):
        o1, S1 = oracle.forward(q, k, v, ones, eta, 1e-3, S0, beta_mode=mode)
        o2, S2 = oracle.forward(q, k, v, None, eta, 1e-3, S0, beta_mode=mode)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(S1, S2)


def test_varlen_and_decode_take_the_mode():
    q, k, v, alpha, eta, S0 = _case(6, T=10)
    o_ref, S_ref = oracle.forward(q, k, v, alpha, eta, 1e-6, S0, beta_mode="given")
    o_v, S_v = oracle.forward_varlen(q[0], k[0], v[0], alpha[0], eta[0], 1e-6, [0, 10], S0,
                                     beta_mode="given")
    np.testing.assert_array_equal(o_v, o_ref[0])
    np.testing.assert_array_equal(S_v, S_ref)
    o_d, S_d = oracle.decode(q[:, 0], k[:, 0], v[:, 0], alpha[:, 0], eta[:, 0], 1e-6, S0,
                             beta_mode="given")
    o_1, S_1 = oracle.forward(q[:, :1], k[:, :1], v[:, :1], alpha[:, :1], eta[:, :1], 1e-6, S0,
                              beta_mode="given")
    np.testing.assert_array_equal(o_d, o_1[:, 0])
    np.testing.assert_array_equal(S_d, S_1)


def test_a_mode_mistake_is_caught(tmp_path):
    """Planted in a copy of the source: the given mode still divides by
    ||k||^2 + eps.  The single-write closed form fails."""
    src = oracle.source()
    bad = src.replace("double beta = et;\n        if (J->beta_mode == 0) {",
                      "double beta = et;\n        if (J->beta_mode >= 0) {")
    assert bad != src
    var = oracle.compile_variant(bad, str(tmp_path / "bad_mode.so"))
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 1, 4)); k = 3.0 * rng.standard_normal((1, 1, 1, 4))
    v = rng.standard_normal((1, 1, 1, 3)); beta = np.full((1, 1, 1), 0.37)
    o, S = var.forward(q, k, v, None, beta, 0.5, None, beta_mode="given")
    assert not np.allclose(S[0, 0], 0.37 * np.outer(k[0, 0, 0], v[0, 0, 0]), rtol=1e-6)
