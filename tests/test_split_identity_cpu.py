"""The sequence-split identity, on the oracle (fp64, CPU).

The recurrence of the Kaczmarz Linear Attention summary (gist.science
2605.08587, "A Regra de Atualizacao KLA") is linear in (V, S0) jointly for
fixed q, k, alpha, eta: beta_t depends on k_t alone.  So a later segment of a
sequence, started from its true state S_s, has

    o   = o(V, 0) + Q_corr S_s,     S_end = N_s + Phi_s S_s,

with o(V, 0), N_s the segment run from a zero state and Q_corr = o(0, I),
Phi_s = S_T(0, I) the same tokens run with V = 0 from the identity.  The split
forward runs the segments side by side on these terms and then chains
S_1 = N_0, S_{s+1} = N_s + Phi_s S_s.  This file checks the identity on the
oracle for segments of unequal length (the split cuts a sequence into whole
128-token tiles as equal as the tile count allows), so a reading error in the
split's algebra fails here without any GPU.
"""
import numpy as np
import pytest

import oracle

D = 32


def _inputs(seed, T):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, D)) / np.sqrt(D)
    k = rng.standard_normal((1, T, 1, D)) / np.sqrt(D) * np.exp(0.5 * rng.standard_normal((1, T, 1, 1)))
    v = rng.standard_normal((1, T, 1, D))
    # decay close to 1 (about 0.996 per token) and weak writes (eta about 0.1),
    # so that a segment's start state still matters at its end: Phi and
    # Q_corr S_s are far from negligible
    alpha = np.exp(-0.005 * np.log1p(np.exp(rng.standard_normal((1, T, 1)))))
    eta = 0.2 / (1.0 + np.exp(-rng.standard_normal((1, T, 1))))
    S0 = rng.standard_normal((1, 1, D, D))
    return q, k, v, alpha, eta, S0


def _seg(x, sl):
    return np.ascontiguousarray(x[:, sl])


def _terms(q, k, v, alpha, eta, eps, sl):
    """(o(V, 0), N, Q_corr, Phi) of the tokens in sl."""
    args = [_seg(x, sl) for x in (q, k, v, alpha, eta)]
    o_v0, N = oracle.forward(*args, eps, None)
    args[2] = np.zeros_like(args[2])
    Qc, Phi = oracle.forward(*args, eps, np.eye(D)[None, None])
    return o_v0[0, :, 0], N[0, 0], Qc[0, :, 0], Phi[0, 0]


def _split_forward(q, k, v, alpha, eta, eps, S0, bounds):
    """The split's terms computed segment by segment with the oracle, then
    chained and corrected; bounds = token offsets [0, b1, ..., T]."""
    sl0 = slice(bounds[0], bounds[1])
    o0, S = oracle.forward(*[_seg(x, sl0) for x in (q, k, v, alpha, eta)], eps, S0)
    outs, S = [o0[0, :, 0]], S[0, 0]
    for s in range(1, len(bounds) - 1):
        o_v0, N, Qc, Phi = _terms(q, k, v, alpha, eta, eps, slice(bounds[s], bounds[s + 1]))
        outs.append(o_v0 + Qc @ S)
        S = N + Phi @ S
    return np.concatenate(outs, axis=0), S


@pytest.mark.parametrize("T,bounds", [
    (640, [0, 384, 640]),                  # 3 + 2 tiles
    (896, [0, 384, 640, 896]),             # 3 + 2 + 2 tiles
    (1152, [0, 256] + [256 + 128 * i for i in range(1, 8)]),   # 2 + 1 x 7 tiles
    (700, [0, 300, 520, 700]),             # not tile-aligned: the identity holds for any cut
])
def test_split_identity_unequal_segments(T, bounds):
    q, k, v, alpha, eta, S0 = _inputs(T, T)
    eps = 1e-6
    o_ref, S_ref = oracle.forward(q, k, v, alpha, eta, eps, S0)
    o_ref, S_ref = o_ref[0, :, 0], S_ref[0, 0]
    o, S = _split_forward(q, k, v, alpha, eta, eps, S0, bounds)
    assert np.abs(o - o_ref).max() <= 1e-10 * np.abs(o_ref).max()
    assert np.abs(S - S_ref).max() <= 1e-10 * np.abs(S_ref).max()


def test_split_terms_matter_and_a_wrong_combine_is_caught():
    """The start state's terms are not negligible here (dropping them, or
    applying Phi on the wrong side, breaks the identity), so the check above
    is not vacuous."""
    T, bounds = 640, [0, 384, 640]
    q, k, v, alpha, eta, S0 = _inputs(7, T)
    eps = 1e-6
    o_ref, S_ref = oracle.forward(q, k, v, alpha, eta, eps, S0)
    S_ref = S_ref[0, 0]
    _, S1 = oracle.forward(*[_seg(x, slice(0, 384)) for x in (q, k, v, alpha, eta)], eps, S0)
    S1 = S1[0, 0]
    _, N, _, Phi = _terms(q, k, v, alpha, eta, eps, slice(384, 640))
    tol = 1e-3 * np.abs(S_ref).max()
    assert np.abs(N + Phi @ S1 - S_ref).max() <= 1e-10 * np.abs(S_ref).max()
    assert np.abs(N - S_ref).max() > tol            # without the start state's term
    assert np.abs(N + S1 @ Phi - S_ref).max() > tol  # Phi on the wrong side
