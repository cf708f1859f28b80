"""The chunkwise-parallel form agrees with the sequential recurrence.

The Kaczmarz Linear Attention summary (gist.science 2605.08587, sections
"Implementacao" and "Contribuicoes Principais" item 2) states that KLA keeps
Gated DeltaNet's chunkwise (blockwise) training algorithm and that the only
change is the diagonal coefficient matrix B = Diag(beta_1..beta_C) inside the
block solver.  The pages print no formulas for that algorithm; the reading
used (and implemented by the CUDA kernels) is the WY/UT form of the delta rule
with B inserted, derived from the recurrence:

    g_i   = sum_{j<=i in chunk} log alpha_j,   Gamma_ij = exp(g_i - g_j)
    T     = (I + B (strict_lower(Gamma o K K^T)))^{-1}
    W     = T B diag(exp g) K,    U~ = T B V,    U = U~ - W S
    O     = diag(exp g) Q S + lower(Gamma o Q K^T) U
    S'    = exp(g_C) S + (diag(exp(g_C - g)) K)^T U

This file restates that form in plain numpy fp64 (a brute-force second
implementation, test only) and checks it against the oracle for several chunk
lengths, including ragged final chunks and the normalised-key rewrite.
"""
import numpy as np
import pytest

import oracle


def chunked_unit(q, k, v, alpha, eta, eps, S0, C, normalise_keys=False, beta_given=False):
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else S0.copy()
    o = np.zeros((T, dv))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        Qc, Kc, Vc = q[sl], k[sl], v[sl]
        n = Qc.shape[0]
        g = np.cumsum(np.log(alpha[sl]))
        n2 = np.sum(Kc * Kc, axis=1)
        den = n2 + eps
        beta = np.where(den == 0, 0.0, eta[sl] / np.where(den == 0, 1.0, den))
        if beta_given:   # Gated DeltaNet: the write strength is eta itself
            beta = eta[sl].copy()
        if normalise_keys:
            # k = |k| k^: beta k e^T = (beta |k|^2) k^ (v/|k| - S~^T k^)^T
            nk = np.sqrt(n2)
            Kc = Kc / nk[:, None]
            Vc = Vc / nk[:, None]
            beta = beta * n2
        diff = g[:, None] - g[None, :]
        Gam = np.exp(np.where(diff <= 0, diff, 0.0))   # only s <= t is used
        Akk = np.tril(Gam * (Kc @ Kc.T), -1)
        Aqk = np.tril(Gam * (Qc @ Kc.T), 0)
        Tm = np.linalg.inv(np.eye(n) + beta[:, None] * Akk)
        W = Tm @ ((beta * np.exp(g))[:, None] * Kc)
        U = Tm @ (beta[:, None] * Vc) - W @ S
        o[sl] = np.exp(g)[:, None] * (Qc @ S) + Aqk @ U
        S = np.exp(g[-1]) * S + (np.exp(g[-1] - g)[:, None] * Kc).T @ U
    return o, S


def _case(seed, T, dk, dv, norm_sigma):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, dk)) / np.sqrt(dk)
    k = rng.standard_normal((1, T, 1, dk)) / np.sqrt(dk) * np.exp(norm_sigma * rng.standard_normal((1, T, 1, 1)))
    v = rng.standard_normal((1, T, 1, dv))
    alpha = 1.0 / (1.0 + np.exp(rng.standard_normal((1, T, 1))))
    eta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, 1))))
    S0 = 0.1 * rng.standard_normal((1, 1, dk, dv))
    return q, k, v, alpha, eta, S0


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16, 64])
@pytest.mark.parametrize("normalise_keys", [False, True])
def test_chunked_equals_sequential(C, normalise_keys):
    T, dk, dv = 75, 8, 6          # 75 = ragged final chunk for every C > 1 here
    q, k, v, alpha, eta, S0 = _case(C, T, dk, dv, 0.5)
    eps = 1e-6
    o_ref, S_ref = oracle.forward(q, k, v, alpha, eta, eps, S0)
    o, S = chunked_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], alpha[0, :, 0], eta[0, :, 0],
                        eps, S0[0, 0], C, normalise_keys)
    scale_o = np.abs(o_ref).max()
    scale_S = np.abs(S_ref).max()
    assert np.abs(o - o_ref[0, :, 0]).max() <= 1e-12 * scale_o
    assert np.abs(S - S_ref[0, 0]).max() <= 1e-12 * scale_S


def test_chunked_equals_sequential_stress_norms():
    """Key norms lognormal(0,1), eta = 1: the over/under-correction regime."""
    T, dk, dv, C = 200, 16, 16, 64
    q, k, v, alpha, eta, S0 = _case(99, T, dk, dv, 1.0)
    eta[:] = 1.0
    o_ref, S_ref = oracle.forward(q, k, v, alpha, eta, 1e-6, S0)
    for nk in (False, True):
        o, S = chunked_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], alpha[0, :, 0], eta[0, :, 0],
                            1e-6, S0[0, 0], C, nk)
        assert np.abs(o - o_ref[0, :, 0]).max() <= 1e-10 * np.abs(o_ref).max()
        assert np.abs(S - S_ref[0, 0]).max() <= 1e-10 * np.abs(S_ref).max()


def test_a_planted_mistake_is_caught():
    """Guard on the guard: a chunk form with the decay applied after the
    residual (a plausible misreading) disagrees with the oracle."""
    T, dk, dv, C = 40, 8, 8, 8
    q, k, v, alpha, eta, S0 = _case(5, T, dk, dv, 0.5)
    o_ref, _ = oracle.forward(q, k, v, alpha, eta, 1e-6, S0)
    # shift alpha by one token: residual against the undecayed state
    alpha_shift = np.concatenate([alpha[:, 1:], alpha[:, :1]], axis=1)
    o, _ = chunked_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], alpha_shift[0, :, 0], eta[0, :, 0],
                        1e-6, S0[0, 0], C)
    assert np.abs(o - o_ref[0, :, 0]).max() > 1e-3 * np.abs(o_ref).max()


@pytest.mark.parametrize("C", [4, 16, 64])
def test_chunked_equals_sequential_given_beta(C):
    """The same block algorithm with B = Diag(beta) for a given beta (Gated
    DeltaNet) matches the oracle's "given" mode."""
    T, dk, dv = 75, 8, 6
    q, k, v, alpha, eta, S0 = _case(40 + C, T, dk, dv, 0.5)
    o_ref, S_ref = oracle.forward(q, k, v, alpha, eta, 1e-6, S0, beta_mode="given")
    o, S = chunked_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], alpha[0, :, 0], eta[0, :, 0],
                        1e-6, S0[0, 0], C, beta_given=True)
    assert np.abs(o - o_ref[0, :, 0]).max() <= 1e-11 * np.abs(o_ref).max()
    assert np.abs(S - S_ref[0, 0]).max() <= 1e-11 * np.abs(S_ref).max()
