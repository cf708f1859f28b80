"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Passages (Kaczmarz Linear Attention summary, gist.science 2605.08587):
  * "Derivacao Teorica": S_t is the state closest (Frobenius) to the decayed
    previous state subject to S^T k_t = v_t; with eta = 1, eps = 0 the step is
    the orthogonal projection, coefficient 1/||k||^2.
  * "A Regra de Atualizacao KLA": beta_t = eta_t/(||k_t||^2 + eps),
    S_t = S~ + beta_t k_t e_t^T, e_t = v_t - S~^T k_t.
  * "Propriedades Chave": orthogonal projection, exact line search,
    normalised gradient step (eta = 1, eps = 0).
Gated DeltaNet gate and the DeltaNet special case: "Linear Attention
Architectures" (gist.science 2607.07953), "Metodologia e Estrutura".
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, T=12, dk=6, dv=5, norm_sigma=1.0, eta_one=False, eps=0.0, s0=True):
    q = rng.standard_normal((1, T, 1, dk))
    k = rng.standard_normal((1, T, 1, dk)) * np.exp(norm_sigma * rng.standard_normal((1, T, 1, 1)))
    v = rng.standard_normal((1, T, 1, dv))
    alpha = rng.uniform(0.3, 1.0, (1, T, 1))
    eta = np.ones((1, T, 1)) if eta_one else rng.uniform(0.05, 1.0, (1, T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv)) if s0 else None
    return q, k, v, alpha, eta, eps, S0


def _states(q, k, v, alpha, eta, eps, S0):
    """Run the oracle one token at a time; returns states S_0..S_T and o."""
    T = q.shape[1]
    dk, dv = q.shape[-1], v.shape[-1]
    S = np.zeros((1, 1, dk, dv)) if S0 is None else S0
    out_S, out_o = [S[0, 0].copy()], []
    for t in range(T):
        o, S = oracle.forward(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1],
                              alpha[:, t:t + 1], eta[:, t:t + 1], eps, S)
        out_S.append(S[0, 0].copy())
        out_o.append(o[0, 0, 0].copy())
    return out_S, np.array(out_o)


def test_chained_single_tokens_equal_one_call():
    rng = np.random.default_rng(1)
    case = _rand_case(rng, eps=1e-3)
    Ss, os_ = _states(*case)
    o, S = oracle.forward(*case)
    np.testing.assert_array_equal(S[0, 0], Ss[-1])
    np.testing.assert_array_equal(o[0, :, 0], os_)


def test_hand_worked_example():
    """Three tokens worked by hand in exact arithmetic (golden fixture)."""
    vals = {}
    with open(os.path.join(GOLDEN, "hand_worked_dk2.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, val = line.split("=")
                vals[key.strip()] = np.array([float(x) for x in val.split()])
    S = vals["S0"].reshape(1, 1, 2, 2)
    for t in (1, 2, 3):
        g = lambda n: vals[f"t{t}.{n}"]
        o, S = oracle.forward(g("q").reshape(1, 1, 1, 2), g("k").reshape(1, 1, 1, 2),
                              g("v").reshape(1, 1, 1, 2), g("alpha").reshape(1, 1, 1),
                              g("eta").reshape(1, 1, 1), float(g("eps")[0]), S)
        np.testing.assert_allclose(S.reshape(-1), g("S"), rtol=0, atol=1e-15)
        np.testing.assert_allclose(o.reshape(-1), g("o"), rtol=0, atol=1e-15)


def test_orthogonal_projection_constraint_holds():
    """eta=1, eps=0: every update satisfies S_t^T k_t = v_t."""
    rng = np.random.default_rng(2)
    q, k, v, alpha, eta, eps, S0 = _rand_case(rng, T=30, eta_one=True, eps=0.0, norm_sigma=1.5)
    Ss, _ = _states(q, k, v, alpha, eta, eps, S0)
    for t in range(q.shape[1]):
        r = Ss[t + 1].T @ k[0, t, 0] - v[0, t, 0]
        assert np.linalg.norm(r) <= 1e-12 * (np.linalg.norm(v[0, t, 0]) + 1e-300) * 10


def test_projection_is_minimum_norm_change():
    """eta=1, eps=0: S_t - S~ is the least-Frobenius-norm correction that
    meets the constraint; compare with numpy's minimum-norm least squares,
    and check that adding any Z with Z^T k = 0 only increases the change."""
    rng = np.random.default_rng(3)
    q, k, v, alpha, eta, eps, S0 = _rand_case(rng, T=10, eta_one=True)
    Ss, _ = _states(q, k, v, alpha, eta, eps, S0)
    for t in range(q.shape[1]):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = alpha[0, t, 0] * Ss[t]
        dS = Ss[t + 1] - St
        # min ||X||_F s.t. X^T k = v - St^T k : one least-norm system per column
        X, *_ = np.linalg.lstsq(kt[None, :], (vt - St.T @ kt)[None, :], rcond=None)
        np.testing.assert_allclose(dS, X, rtol=1e-11, atol=1e-12)
        Z = rng.standard_normal(dS.shape)
        Z -= np.outer(kt, kt @ Z) / (kt @ kt)     # Z^T k = 0
        assert np.linalg.norm(dS + Z) > np.linalg.norm(dS)
        np.testing.assert_allclose((St + dS + Z).T @ kt, vt, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("eta_one,eps", [(True, 0.0), (False, 0.0), (False, 0.3)])
def test_exact_line_search(eta_one, eps):
    """The step taken along k e^T is the exact minimiser of the per-token loss
    phi(s) = 1/2 ||(S~ + s k e^T)^T k - v||^2 (found by scipy), scaled by
    eta ||k||^2/(||k||^2 + eps) when relaxed."""
    from scipy.optimize import minimize_scalar
    rng = np.random.default_rng(4)
    q, k, v, alpha, eta, _, S0 = _rand_case(rng, T=8, eta_one=eta_one)
    Ss, _ = _states(q, k, v, alpha, eta, eps, S0)
    for t in range(q.shape[1]):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = alpha[0, t, 0] * Ss[t]
        e = vt - St.T @ kt
        D = np.outer(kt, e)
        dS = Ss[t + 1] - St
        s_taken = np.sum(dS * D) / np.sum(D * D)
        np.testing.assert_allclose(dS, s_taken * D, rtol=1e-11, atol=1e-13)
        phi = lambda s: 0.5 * np.sum(((St + s * D).T @ kt - vt) ** 2)
        n2 = kt @ kt
        res = minimize_scalar(phi, bracket=(0.0, 2.0 / n2), tol=1e-14)
        relax = eta[0, t, 0] * n2 / (n2 + eps)
        np.testing.assert_allclose(s_taken, relax * res.x, rtol=1e-6)
        if eta_one and eps == 0.0:
            assert phi(s_taken) <= 1e-20 * max(1.0, e @ e)
            for d in (1e-3, 0.1):
                assert phi(s_taken * (1 + d)) > phi(s_taken)
                assert phi(s_taken * (1 - d)) > phi(s_taken)


def test_normalised_gradient_step():
    """eta=1, eps=0: S_t - S~ = -(1/||k||^2) grad L(S~), L(S) = 1/2||S^T k - v||^2,
    with the gradient taken by central finite differences."""
    rng = np.random.default_rng(5)
    q, k, v, alpha, eta, eps, S0 = _rand_case(rng, T=5, dk=4, dv=3, eta_one=True)
    Ss, _ = _states(q, k, v, alpha, eta, eps, S0)
    for t in range(q.shape[1]):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = alpha[0, t, 0] * Ss[t]
        L = lambda S: 0.5 * np.sum((S.T @ kt - vt) ** 2)
        G = np.zeros_like(St)
        h = 1e-6
        for i in range(St.shape[0]):
            for j in range(St.shape[1]):
                E = np.zeros_like(St)
                E[i, j] = h
                G[i, j] = (L(St + E) - L(St - E)) / (2 * h)
        np.testing.assert_allclose(Ss[t + 1] - St, -G / (kt @ kt), rtol=1e-6, atol=1e-8)


def test_residual_closed_form_any_eta_eps():
    """For every token, S_t^T k_t - v_t = -(1 - eta n^2/(n^2+eps)) e_t with
    e_t = v_t - alpha_t S_{t-1}^T k_t: decay before residual, current alpha,
    eps added once to ||k||^2."""
    rng = np.random.default_rng(6)
    q, k, v, alpha, eta, _, S0 = _rand_case(rng, T=20)
    eps = 0.7
    Ss, _ = _states(q, k, v, alpha, eta, eps, S0)
    for t in range(q.shape[1]):
        kt, vt = k[0, t, 0], v[0, t, 0]
        e = vt - alpha[0, t, 0] * Ss[t].T @ kt
        n2 = kt @ kt
        lhs = Ss[t + 1].T @ kt - vt
        np.testing.assert_allclose(lhs, -(1 - eta[0, t, 0] * n2 / (n2 + eps)) * e,
                                   rtol=1e-10, atol=1e-12)


def test_decay_only_when_eta_zero():
    rng = np.random.default_rng(7)
    q, k, v, alpha, _, eps, S0 = _rand_case(rng, T=15, eps=1e-6)
    eta = np.zeros_like(alpha)
    o, S = oracle.forward(q, k, v, alpha, eta, eps, S0)
    P = np.cumprod(alpha[0, :, 0])
    np.testing.assert_allclose(S[0, 0], P[-1] * S0[0, 0], rtol=1e-13)
    for t in range(q.shape[1]):
        np.testing.assert_allclose(o[0, t, 0], P[t] * S0[0, 0].T @ q[0, t, 0], rtol=1e-12, atol=1e-14)


def test_single_write_from_zero_state():
    rng = np.random.default_rng(8)
    dk, dv = 7, 5
    q = rng.standard_normal((1, 1, 1, dk)); k = rng.standard_normal((1, 1, 1, dk))
    v = rng.standard_normal((1, 1, 1, dv))
    alpha = np.ones((1, 1, 1)); eta = np.full((1, 1, 1), 0.37); eps = 0.25
    o, S = oracle.forward(q, k, v, alpha, eta, eps, None)
    kt, qt, vt = k[0, 0, 0], q[0, 0, 0], v[0, 0, 0]
    beta = 0.37 / (kt @ kt + eps)
    np.testing.assert_allclose(S[0, 0], beta * np.outer(kt, vt), rtol=1e-13)
    np.testing.assert_allclose(o[0, 0, 0], beta * (kt @ qt) * vt, rtol=1e-13)


def test_orthogonal_keys_overwrite_rows():
    """k_t = c_t e_{i_t} with distinct i_t, alpha=1, eta=1, eps=0: row i_t of
    S_T is v_t / c_t and untouched rows keep S0."""
    rng = np.random.default_rng(9)
    dk, dv, T = 8, 4, 5
    idx = rng.permutation(dk)[:T]
    c = rng.uniform(0.2, 5.0, T) * rng.choice([-1, 1], T)
    k = np.zeros((1, T, 1, dk))
    for t in range(T):
        k[0, t, 0, idx[t]] = c[t]
    v = rng.standard_normal((1, T, 1, dv)); q = rng.standard_normal((1, T, 1, dk))
    S0 = rng.standard_normal((1, 1, dk, dv))
    o, S = oracle.forward(q, k, v, np.ones((1, T, 1)), np.ones((1, T, 1)), 0.0, S0)
    for t in range(T):
        np.testing.assert_allclose(S[0, 0, idx[t]], v[0, t, 0] / c[t], rtol=1e-14)
    for i in set(range(dk)) - set(idx.tolist()):
        np.testing.assert_array_equal(S[0, 0, i], S0[0, 0, i])


def test_zero_key_with_zero_eps_writes_nothing():
    rng = np.random.default_rng(10)
    q, k, v, alpha, eta, _, S0 = _rand_case(rng, T=3)
    k[0, 1] = 0.0
    Ss, os_ = _states(q, k, v, alpha, eta, 0.0, S0)
    np.testing.assert_allclose(Ss[2], alpha[0, 1, 0] * Ss[1], rtol=1e-15)
    assert np.all(np.isfinite(os_))


def test_gated_deltanet_reduction_unit_keys():
    """Unit-norm keys and eps=0 reduce KLA to Gated DeltaNet with beta = eta.
    Gated DeltaNet here is written in its (dv x dk) transition form
    M_t = alpha_t M_{t-1} (I - b_t k k^T) + b_t v k^T, read o = M q."""
    rng = np.random.default_rng(11)
    T, dk, dv = 16, 6, 4
    q, k, v, alpha, eta, _, S0 = _rand_case(rng, T=T, dk=dk, dv=dv)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o, S = oracle.forward(q, k, v, alpha, eta, 0.0, S0)
    M = S0[0, 0].T.copy()
    for t in range(T):
        kt, b = k[0, t, 0], eta[0, t, 0]
        M = alpha[0, t, 0] * M @ (np.eye(dk) - b * np.outer(kt, kt)) + b * np.outer(v[0, t, 0], kt)
        np.testing.assert_allclose(o[0, t, 0], M @ q[0, t, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S[0, 0], M.T, rtol=1e-12, atol=1e-13)


def test_deltanet_special_case_alpha_one():
    """alpha = 1 is DeltaNet (residual write, no decay): the state after a
    repeated identical (k, v) with eta = 1, eps = 0 is unchanged by the repeat."""
    rng = np.random.default_rng(12)
    dk, dv = 5, 3
    kt = rng.standard_normal(dk); vt = rng.standard_normal(dv)
    k = np.stack([kt, kt])[None, :, None]; v = np.stack([vt, vt])[None, :, None]
    q = rng.standard_normal((1, 2, 1, dk))
    S0 = rng.standard_normal((1, 1, dk, dv))
    Ss, _ = _states(q, k, v, np.ones((1, 2, 1)), np.ones((1, 2, 1)), 0.0, S0)
    np.testing.assert_allclose(Ss[2], Ss[1], rtol=1e-13, atol=1e-14)


def test_stability_bound():
    """eta in [0,1], eps >= 0: ||S_t||_2 <= alpha_t ||S_{t-1}||_2 + eta ||v||/||k||."""
    rng = np.random.default_rng(13)
    q, k, v, alpha, eta, _, S0 = _rand_case(rng, T=40, norm_sigma=2.0)
    Ss, _ = _states(q, k, v, alpha, eta, 1e-3, S0)
    for t in range(q.shape[1]):
        lhs = np.linalg.norm(Ss[t + 1], 2)
        rhs = alpha[0, t, 0] * np.linalg.norm(Ss[t], 2) + \
            eta[0, t, 0] * np.linalg.norm(v[0, t, 0]) / np.linalg.norm(k[0, t, 0])
        assert lhs <= rhs * (1 + 1e-12)


def test_transition_matrix_form():
    """S_t = A_t S_{t-1} + beta_t k_t v_t^T with A_t = alpha_t (I - beta_t k_t k_t^T)."""
    rng = np.random.default_rng(14)
    q, k, v, alpha, eta, _, S0 = _rand_case(rng, T=25)
    eps = 0.05
    o, S = oracle.forward(q, k, v, alpha, eta, eps, S0)
    X = S0[0, 0].copy()
    dk = X.shape[0]
    for t in range(q.shape[1]):
        kt = k[0, t, 0]
        b = eta[0, t, 0] / (kt @ kt + eps)
        X = alpha[0, t, 0] * (np.eye(dk) - b * np.outer(kt, kt)) @ X + b * np.outer(kt, v[0, t, 0])
        np.testing.assert_allclose(o[0, t, 0], X.T @ q[0, t, 0], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], X, rtol=1e-11, atol=1e-12)


def test_batch_heads_are_independent_and_layout():
    """Each (b, h) is its own recurrence; [B,T,H,d] rows and [B,H,dk,dv] states
    are indexed as documented (single-unit calls on slices agree)."""
    rng = np.random.default_rng(15)
    B, T, H, dk, dv = 2, 9, 3, 4, 5
    q = rng.standard_normal((B, T, H, dk)); k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv)); alpha = rng.uniform(0.5, 1, (B, T, H))
    eta = rng.uniform(0, 1, (B, T, H)); S0 = rng.standard_normal((B, H, dk, dv))
    o, S = oracle.forward(q, k, v, alpha, eta, 1e-4, S0, nthreads=3)
    for b in range(B):
        for h in range(H):
            o1, S1 = oracle.forward(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1],
                                    v[b:b + 1, :, h:h + 1], alpha[b:b + 1, :, h:h + 1],
                                    eta[b:b + 1, :, h:h + 1], 1e-4, S0[b:b + 1, h:h + 1])
            np.testing.assert_array_equal(o[b, :, h], o1[0, :, 0])
            np.testing.assert_array_equal(S[b, h], S1[0, 0])


def test_varlen_equals_per_sequence_calls():
    rng = np.random.default_rng(16)
    lens = [5, 1, 0, 12, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    H, dk, dv = 2, 4, 3
    tot = int(cu[-1])
    q = rng.standard_normal((tot, H, dk)); k = rng.standard_normal((tot, H, dk))
    v = rng.standard_normal((tot, H, dv)); alpha = rng.uniform(0.5, 1, (tot, H))
    eta = rng.uniform(0, 1, (tot, H)); S0 = rng.standard_normal((len(lens), H, dk, dv))
    o, S = oracle.forward_varlen(q, k, v, alpha, eta, 1e-3, cu, S0, nthreads=2)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        o1, S1 = oracle.forward(q[None, a:b], k[None, a:b], v[None, a:b], alpha[None, a:b],
                                eta[None, a:b], 1e-3, S0[n:n + 1])
        np.testing.assert_array_equal(o[a:b], o1[0])
        np.testing.assert_array_equal(S[n], S1[0])


def test_decode_is_one_token_forward():
    rng = np.random.default_rng(17)
    B, H, dk, dv = 3, 2, 4, 4
    q = rng.standard_normal((B, H, dk)); k = rng.standard_normal((B, H, dk))
    v = rng.standard_normal((B, H, dv)); alpha = rng.uniform(0.5, 1, (B, H))
    eta = rng.uniform(0, 1, (B, H)); S = rng.standard_normal((B, H, dk, dv))
    o, S1 = oracle.decode(q, k, v, alpha, eta, 1e-6, S)
    for b in range(B):
        for h in range(H):
            kt = k[b, h]
            beta = eta[b, h] / (kt @ kt + 1e-6)
            St = alpha[b, h] * S[b, h]
            e = v[b, h] - St.T @ kt
            np.testing.assert_allclose(S1[b, h], St + beta * np.outer(kt, e), rtol=1e-13)
            np.testing.assert_allclose(o[b, h], S1[b, h].T @ q[b, h], rtol=1e-12)
