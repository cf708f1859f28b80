"""The pins have teeth: plausible mistakes planted in a copy of the oracle's C
source (on the CPU) each fail at least one pin, while the real oracle passes
them all.  The pins used here are the hand-worked example, the orthogonal
projection property, the residual closed form for any eta and eps (KLA
summary, gist.science 2605.08587: "Derivacao Teorica", "A Regra de
Atualizacao KLA", "Propriedades Chave"), and the Gated DeltaNet reduction
with unit keys (Linear Attention Architectures, gist.science 2607.07953)."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_dk2.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = np.array([float(x) for x in v.split()])
    return vals


def _pin_hand_worked(orc):
    g = _golden()
    S = g["S0"].reshape(1, 1, 2, 2)
    for t in (1, 2, 3):
        f = lambda n: g[f"t{t}.{n}"]
        o, S = orc.forward(f("q").reshape(1, 1, 1, 2), f("k").reshape(1, 1, 1, 2),
                           f("v").reshape(1, 1, 1, 2), f("alpha").reshape(1, 1, 1),
                           f("eta").reshape(1, 1, 1), float(f("eps")[0]), S)
        if not (np.allclose(S.reshape(-1), f("S"), atol=1e-14) and
                np.allclose(o.reshape(-1), f("o"), atol=1e-14)):
            return False
    return True


def _case(seed, T=10, dk=5, dv=4, eta_one=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, dk)); k = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv)); alpha = rng.uniform(0.3, 1.0, (1, T, 1))
    eta = np.ones((1, T, 1)) if eta_one else rng.uniform(0.1, 1.0, (1, T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv))
    return q, k, v, alpha, eta, S0


def _steps(orc, q, k, v, alpha, eta, eps, S0):
    Ss = [S0[0, 0]]
    S = S0
    for t in range(q.shape[1]):
        _, S = orc.forward(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], alpha[:, t:t + 1],
                           eta[:, t:t + 1], eps, S)
        Ss.append(S[0, 0])
    return Ss


def _pin_projection(orc):
    q, k, v, alpha, eta, S0 = _case(1, eta_one=True)
    Ss = _steps(orc, q, k, v, alpha, eta, 0.0, S0)
    return all(np.allclose(Ss[t + 1].T @ k[0, t, 0], v[0, t, 0], atol=1e-10)
               for t in range(q.shape[1]))


def _pin_residual(orc):
    q, k, v, alpha, eta, S0 = _case(2)
    eps = 0.7
    Ss = _steps(orc, q, k, v, alpha, eta, eps, S0)
    for t in range(q.shape[1]):
        kt, vt = k[0, t, 0], v[0, t, 0]
        e = vt - alpha[0, t, 0] * Ss[t].T @ kt
        n2 = kt @ kt
        if not np.allclose(Ss[t + 1].T @ kt - vt, -(1 - eta[0, t, 0] * n2 / (n2 + eps)) * e,
                           atol=1e-10):
            return False
    return True


def _pin_gdn(orc):
    q, k, v, alpha, eta, S0 = _case(3, dk=5, dv=3)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o, S = orc.forward(q, k, v, alpha, eta, 0.0, S0)
    M = S0[0, 0].T.copy()
    for t in range(q.shape[1]):
        kt, b = k[0, t, 0], eta[0, t, 0]
        M = alpha[0, t, 0] * M @ (np.eye(5) - b * np.outer(kt, kt)) + b * np.outer(v[0, t, 0], kt)
        if not np.allclose(o[0, t, 0], M @ q[0, t, 0], atol=1e-10):
            return False
    return np.allclose(S[0, 0], M.T, atol=1e-10)


PINS = [_pin_hand_worked, _pin_projection, _pin_residual, _pin_gdn]

MUTANTS = {
    "eps_squared": ("const double den = n2 + J->eps;", "const double den = n2 + J->eps * J->eps;"),
    "eta_dropped": ("et / den", "1.0 / den"),
    "norm_not_squared": ("n2 += kt[i] * kt[i];", "n2 += (kt[i] < 0 ? -kt[i] : kt[i]);"),
    "residual_undecayed": ("acc += St[(size_t)i * dv + j] * kt[i];",
                           "acc += S[(size_t)i * dv + j] * kt[i];"),
    "update_sign": ("St[(size_t)i * dv + j] + beta * kt[i] * e[j]",
                    "St[(size_t)i * dv + j] - beta * kt[i] * e[j]"),
    "read_before_write": ("acc += S[(size_t)i * dv + j] * qt[i];",
                          "acc += St[(size_t)i * dv + j] * qt[i];"),
    "read_transposed": ("acc += S[(size_t)i * dv + j] * qt[i];",
                        "acc += S[(size_t)j * dv + i] * qt[i];"),
    "decay_not_applied": ("St[x] = a * S[x];", "St[x] = S[x];"),
}


def test_real_oracle_passes_every_pin():
    class Real:
        forward = staticmethod(oracle.forward)
    assert all(pin(Real) for pin in PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    variant = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    results = [pin(variant) for pin in PINS]
    assert not all(results), f"mutant {name} passed every pin"
