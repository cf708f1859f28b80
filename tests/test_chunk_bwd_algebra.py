"""The chunk form of the backward pass that the CUDA kernels implement,
written out in numpy (fp64), equals the sequential adjoint of the oracle.
This pins the chunk-level derivation (reverse-mode differentiation of the
blockwise solver of the KLA summary, gist.science 2605.08587,
"Implementacao": T = (I + strict_lower(diag(beta) Gamma o K K^T))^-1,
U = T diag(beta) (V - diag(exp g) K S), O = diag(exp g) Q S + lower(Gamma o
Q K^T) U, S' = exp(g_C) S + (diag(exp(g_C - g)) K)^T U) for several chunk
lengths, partial chunks, both write-coefficient modes and eps = 0.

Backward of one chunk, given dO and dS' (the gradient of the state at the
chunk's end):
  dU  = A_qk^T dO + diag(exp(g_C - g)) K dS'
  dR  = T^T dU                      (R = diag(beta)(V - diag(exp g) K S))
  dS  = exp(g_C) dS' + Q^T diag(exp g) dO - K^T diag(beta exp g) dR
  dV  = diag(beta) dR
  dA_kk = -strict_lower(dR U^T),   dA_qk = lower(dO U^T)
and the terms of dQ, dK, dbeta, dg collected below; dlog(alpha) is the
reverse cumulative sum of dg and beta = eta / (||k||^2 + eps) is chained last.
"""
import numpy as np
import pytest

import oracle


def chunk_bwd(q, k, v, alpha, eta, eps, S0, do, dST, C=8, mode=0):
    # single unit: q,k [T,dk], v,do [T,dv], alpha, eta [T]
    T, dk = q.shape; dv = v.shape[1]
    nch = (T + C - 1) // C
    pad = nch * C - T
    P = lambda x, val=0.0: np.concatenate([x, np.full((pad,) + x.shape[1:], val)]) if pad else x
    q, k, v, do = P(q), P(k), P(v), P(do)
    alpha = P(alpha, 1.0); eta = P(eta, 0.0)
    # forward: states at chunk starts
    Ss = []
    S = S0.copy()
    pre = []
    for c in range(nch):
        sl = slice(c*C, (c+1)*C)
        K, Q, V = k[sl], q[sl], v[sl]
        g = np.cumsum(np.log(alpha[sl])); eg = np.exp(g); gC = g[-1]; egc = np.exp(gC - g)
        n2 = (K*K).sum(1); den = n2 + eps
        beta = eta[sl] if mode else np.where(den != 0, eta[sl] / np.where(den != 0, den, 1), 0)
        Gam = np.tril(np.exp(g[:, None] - g[None, :]))
        Gkk = K @ K.T
        Akk = np.tril(beta[:, None] * Gam * Gkk, -1)
        Tm = np.linalg.inv(np.eye(C) + Akk)
        Aqk = Gam * (Q @ K.T)
        pre.append(dict(K=K, Q=Q, V=V, g=g, eg=eg, gC=gC, egc=egc, n2=n2, den=den, beta=beta, Gam=Gam,
                        Gkk=Gkk, Akk=Akk, Tm=Tm, Aqk=Aqk, eta=eta[sl], alpha=alpha[sl]))
        Ss.append(S.copy())
        KS = K @ S; R = beta[:, None] * (V - eg[:, None] * KS); U = Tm @ R
        S = np.exp(gC) * S + (egc[:, None] * K).T @ U
    # backward
    dS = dST.copy()
    dq = np.zeros_like(q); dkk = np.zeros_like(k); dvv = np.zeros_like(v)
    da = np.zeros(nch*C); de = np.zeros(nch*C)
    for c in reversed(range(nch)):
        sl = slice(c*C, (c+1)*C)
        p = pre[c]; S = Ss[c]; dSp = dS
        K, Q, V, g, eg, gC, egc, beta, Gam, Gkk, Akk, Tm, Aqk = (p[x] for x in
            'K Q V g eg gC egc beta Gam Gkk Akk Tm Aqk'.split())
        dO = do[sl]
        KS = K @ S; VmKS = V - eg[:, None] * KS; R = beta[:, None] * VmKS; U = Tm @ R
        dU = Aqk.T @ dO + (egc[:, None] * K) @ dSp
        dR = Tm.T @ dU
        dS = np.exp(gC) * dSp + Q.T @ (eg[:, None] * dO) - K.T @ ((beta * eg)[:, None] * dR)
        dV = beta[:, None] * dR
        dbeta = (VmKS * dR).sum(1)
        dK = -((beta * eg)[:, None] * dR) @ S.T
        dg = -beta * eg * (KS * dR).sum(1)
        dAkk = -np.tril(dR @ U.T, -1)
        dA = np.tril(dO @ U.T)
        dAg = dA * Gam
        QS = Q @ S
        dQ = eg[:, None] * (dO @ S.T) + dAg @ K
        dK += dAg.T @ Q
        X = dAkk * Gam
        bX = beta[:, None] * X
        dK += bX @ K + bX.T @ K
        dbeta += (X * Gkk).sum(1)
        t1 = dAkk * Akk; dg += t1.sum(1) - t1.sum(0)
        t2 = dA * Aqk; dg += t2.sum(1) - t2.sum(0)
        dg += eg * (QS * dO).sum(1)
        dKt = U @ dSp.T
        dK += egc[:, None] * dKt
        w = egc * (K * dKt).sum(1)
        dg -= w
        dgC = w.sum() + np.exp(gC) * (dSp * S).sum()
        dg[-1] += dgC
        dlg = np.cumsum(dg[::-1])[::-1]
        da[sl] = dlg / p['alpha']
        if mode:
            de[sl] = dbeta
        else:
            ok = p['den'] != 0
            de[sl] = np.where(ok, dbeta / np.where(ok, p['den'], 1), 0)
            dK += np.where(ok, -2 * p['eta'] * dbeta / np.where(ok, p['den'], 1)**2, 0)[:, None] * K
        dq[sl] = dQ; dkk[sl] = dK; dvv[sl] = dV
    return dq[:T], dkk[:T], dvv[:T], da[:T], de[:T], dS



@pytest.mark.parametrize("T,dk,dv,C,mode,eps", [
    (21, 5, 4, 8, 0, 0.1), (16, 3, 6, 8, 1, 0.0), (64, 8, 8, 16, 0, 1e-6), (7, 4, 4, 8, 0, 0.0),
    (40, 6, 5, 8, 0, 0.5), (130, 4, 4, 64, 0, 1e-6)])
def test_chunk_backward_equals_sequential_adjoint(T, dk, dv, C, mode, eps):
    rng = np.random.default_rng(T + C)
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk)) * np.exp(rng.standard_normal((T, 1)) * .5)
    v = rng.standard_normal((T, dv)); alpha = rng.uniform(0.3, 1, T); eta = rng.uniform(0.1, 1, T)
    S0 = rng.standard_normal((dk, dv)); do = rng.standard_normal((T, dv))
    dST = rng.standard_normal((dk, dv))
    got = chunk_bwd(q, k, v, alpha, eta, eps, S0, do, dST, C=C, mode=mode)
    ref = oracle.backward(q[None, :, None], k[None, :, None], v[None, :, None],
                          alpha[None, :, None], eta[None, :, None], eps, S0[None, None],
                          do[None, :, None], dST[None, None],
                          beta_mode=["kaczmarz", "given"][mode])
    refs = [ref[0][0, :, 0], ref[1][0, :, 0], ref[2][0, :, 0], ref[3][0, :, 0],
            ref[4][0, :, 0], ref[5][0, 0]]
    for a, b in zip(got, refs):
        assert np.abs(a - b).max() <= 1e-12 * np.abs(b).max()
