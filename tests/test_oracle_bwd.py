"""Pins of the backward oracle (oracle/kla_oracle_bwd.c), none of which reuses
its arithmetic:

* central finite differences of the forward oracle along random directions,
  for every input (q, k, v, alpha, eta, S0), both write-coefficient modes,
  eps > 0 and eps = 0, no decay, no initial state;
* Euler's identity for functions homogeneous of degree one: o and S_T are
  linear in (v, S0) jointly and o is linear in q, so <dv, v> + <dS0, S0> = L
  and <dq, q> = sum <do, o>;
* the closed form of a single token (T = 1), derived by hand from the update
  rule (KLA summary, gist.science 2605.08587, "A Regra de Atualizacao KLA");
* planted mistakes in a copy of the C source each fail a pin.
"""
import numpy as np
import pytest

import oracle


def _case(seed, B=1, T=9, H=2, dk=5, dv=4, eta_scale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk)) * np.exp(0.5 * rng.standard_normal((B, T, H, 1)))
    v = rng.standard_normal((B, T, H, dv))
    alpha = rng.uniform(0.3, 1.0, (B, T, H))
    eta = eta_scale * rng.uniform(0.1, 1.0, (B, T, H))
    S0 = rng.standard_normal((B, H, dk, dv))
    do = rng.standard_normal((B, T, H, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    return q, k, v, alpha, eta, S0, do, dST


def _loss(args, eps, do, dST, mode):
    q, k, v, alpha, eta, S0 = args
    o, S = oracle.forward(q, k, v, alpha, eta, eps, S0, beta_mode=mode)
    L = float((o * do).sum())
    if dST is not None:
        L += float((S * dST).sum())
    return L


def _fd_errors(orc, seed, eps, mode, no_alpha=False, no_S0=False, no_dST=False):
    q, k, v, alpha, eta, S0, do, dST = _case(seed)
    if no_alpha:
        alpha = None
    if no_S0:
        S0 = None
    if no_dST:
        dST = None
    g = orc.backward(q, k, v, alpha, eta, eps, S0, do, dST, beta_mode=mode)
    args = [q, k, v, alpha, eta, S0]
    rng = np.random.default_rng(seed + 100)
    errs = {}
    for i, name in enumerate(["q", "k", "v", "alpha", "eta", "S0"]):
        if args[i] is None:
            continue
        d = rng.standard_normal(args[i].shape)
        h = 1e-6
        ap = list(args); ap[i] = args[i] + h * d
        am = list(args); am[i] = args[i] - h * d
        fd = (_loss(ap, eps, do, dST, mode) - _loss(am, eps, do, dST, mode)) / (2 * h)
        an = float((g[i] * d).sum())
        errs[name] = abs(fd - an) / max(1e-9, abs(fd))
    return errs


@pytest.mark.parametrize("eps,mode,no_alpha,no_S0,no_dST", [
    (1e-6, "kaczmarz", False, False, False), (0.0, "kaczmarz", False, False, False),
    (0.7, "kaczmarz", False, True, True), (0.0, "given", False, False, False),
    (0.1, "kaczmarz", True, False, False), (0.1, "given", True, True, False)])
def test_gradient_matches_finite_differences(eps, mode, no_alpha, no_S0, no_dST):
    class Real:
        backward = staticmethod(oracle.backward)
    errs = _fd_errors(Real, 3, eps, mode, no_alpha, no_S0, no_dST)
    assert max(errs.values()) < 1e-6, errs


@pytest.mark.parametrize("mode", ["kaczmarz", "given"])
def test_euler_identities(mode):
    q, k, v, alpha, eta, S0, do, dST = _case(4, T=70)
    dq, dk, dv, da, de, dS0 = oracle.backward(q, k, v, alpha, eta, 0.2, S0, do, dST,
                                              beta_mode=mode)
    o, S = oracle.forward(q, k, v, alpha, eta, 0.2, S0, beta_mode=mode)
    L = (o * do).sum() + (S * dST).sum()
    assert abs((dv * v).sum() + (dS0 * S0).sum() - L) <= 1e-10 * abs(L)
    Lo = (o * do).sum()
    assert abs((dq * q).sum() - Lo) <= 1e-10 * abs(Lo)


def test_single_token_closed_form():
    rng = np.random.default_rng(5)
    dk, dv, eps = 4, 3, 0.3
    q, k = rng.standard_normal((2, dk)); v = rng.standard_normal(dv)
    a, eta = 0.8, 0.6
    S0 = rng.standard_normal((dk, dv)); do = rng.standard_normal(dv)
    n2 = k @ k; den = n2 + eps; beta = eta / den
    P = np.eye(dk) - beta * np.outer(k, k)
    S1 = a * P @ S0 + beta * np.outer(k, v)
    e = v - a * S0.T @ k
    dq = S1 @ do
    dval = beta * (k @ q) * do
    dS0 = a * np.outer(P @ q, do)
    dalpha = q @ P @ S0 @ do
    dbeta = (k @ q) * (e @ do)
    deta = dbeta / den
    dk_ = (beta * (v @ do) * q - a * beta * ((k @ S0 @ do) * q + (q @ k) * (S0 @ do))
           - 2 * eta * dbeta / den ** 2 * k)
    g = oracle.backward(q.reshape(1, 1, 1, dk), k.reshape(1, 1, 1, dk), v.reshape(1, 1, 1, dv),
                        np.full((1, 1, 1), a), np.full((1, 1, 1), eta), eps,
                        S0.reshape(1, 1, dk, dv), do.reshape(1, 1, 1, dv))
    for got, want in zip(g, [dq, dk_, dval, dalpha, deta, dS0]):
        np.testing.assert_allclose(np.asarray(got).reshape(-1), np.asarray(want).reshape(-1),
                                   rtol=1e-12, atol=1e-13)


MUTANTS = {
    "read_grad_transposed": ("acc += S[(size_t)i * dv + j] * dot[j];",
                             "acc += S[(size_t)i * dv + j] * dot[i % dv];"),
    "beta_term_dropped": ("dbeta += kt[i] * dse;", "dbeta += 0.0 * dse;"),
    "residual_sign": ("dkt[i] -= acc;", "dkt[i] += acc;"),
    "decay_adjoint_missing": ("dS[x] = a * dSt[x];", "dS[x] = dSt[x];"),
    "norm_chain_factor": ("const double c = -2.0 * et * dbeta / (den * den);",
                          "const double c = -1.0 * et * dbeta / (den * den);"),
    "dalpha_on_new_state": ("da += dSt[x] * Sp[x];", "da += dSt[x] * S[x];"),
    "dv_unscaled": ("de[j] = beta * acc;", "de[j] = acc;"),
}


def test_real_backward_passes_the_pins():
    class Real:
        backward = staticmethod(oracle.backward)
    assert max(_fd_errors(Real, 7, 0.2, "kaczmarz").values()) < 1e-6


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_backward_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_bwd()
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    variant = oracle.compile_bwd_variant(src.replace(old, new), str(tmp_path / f"bm_{name}.so"))
    errs = _fd_errors(variant, 7, 0.2, "kaczmarz")
    assert max(errs.values()) > 1e-4, f"mutant {name} passed: {errs}"
