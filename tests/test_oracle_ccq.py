"""Pins for the CCQ oracle (CPU): the Curvature-Conditioned Query of "Don't
Read Everything: A Curvature-Conditioned Query for Linear Attention"
(gist.science 2606.01294), q_clean_t = (I - lambda_t Sigma_t) q_t with
Sigma_t = Cov_{<=t}[k] ("Derivacao Teorica", "O Mecanismo"), read against the
unchanged recurrence ("Integracao")."""
import numpy as np

import oracle


def _keys(seed, T=11, dk=5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, dk))
    k = rng.standard_normal((1, T, 1, dk)) + 0.3
    lam = rng.uniform(0.0, 1.0, (1, T, 1))
    return q, k, lam


def test_covariance_is_numpys_population_covariance():
    q, k, lam = _keys(1)
    qc, _ = oracle.ccq_query(q, k, lam)
    K = k[0, :, 0]
    for t in range(K.shape[0]):
        Sig = np.cov(K[:t + 1].T, bias=True) if t > 0 else np.zeros((5, 5))
        np.testing.assert_allclose(qc[0, t, 0], q[0, t, 0] - lam[0, t, 0] * Sig @ q[0, t, 0],
                                   rtol=1e-12, atol=1e-13)


def test_zero_gate_and_constant_keys_leave_the_query():
    q, k, lam = _keys(2)
    qc, _ = oracle.ccq_query(q, k, np.zeros_like(lam))
    np.testing.assert_array_equal(qc, q)
    kc = np.broadcast_to(k[:, :1], k.shape).copy()   # every key the same: Sigma = 0
    qc, _ = oracle.ccq_query(q, kc, lam)
    np.testing.assert_allclose(qc, q, rtol=0, atol=1e-13)


def test_keys_on_one_axis_closed_form():
    """k_j = c_j e_1: Sigma_t = Var(c_<=t) e_1 e_1^T, so only the e_1 part of
    the query shrinks, by lambda_t Var(c_<=t)."""
    rng = np.random.default_rng(3)
    T, dk = 9, 4
    c = rng.standard_normal(T) * 2.0
    k = np.zeros((1, T, 1, dk)); k[0, :, 0, 0] = c
    q = rng.standard_normal((1, T, 1, dk)); lam = rng.uniform(0, 1, (1, T, 1))
    qc, _ = oracle.ccq_query(q, k, lam)
    for t in range(T):
        want = q[0, t, 0].copy()
        want[0] *= 1.0 - lam[0, t, 0] * np.var(c[:t + 1])
        np.testing.assert_allclose(qc[0, t, 0], want, rtol=1e-12, atol=1e-13)


def test_statistics_carry_across_calls():
    q, k, lam = _keys(4, T=12)
    qc, st = oracle.ccq_query(q, k, lam)
    qa, sa = oracle.ccq_query(q[:, :5], k[:, :5], lam[:, :5])
    qb, sb = oracle.ccq_query(q[:, 5:], k[:, 5:], lam[:, 5:], stats0=sa)
    np.testing.assert_allclose(np.concatenate([qa, qb], 1), qc, rtol=1e-12, atol=1e-13)
    for x, y in zip(sb, st):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)
    assert st[2][0, 0] == 12.0


def test_ccq_read_of_a_fixed_state():
    """No writes (eta = 0, alpha = 1): the CCQ output is S0^T q_clean."""
    q, k, lam = _keys(5, T=6, dk=4)
    rng = np.random.default_rng(6)
    S0 = rng.standard_normal((1, 1, 4, 3))
    v = rng.standard_normal((1, 6, 1, 3))
    qc, _ = oracle.ccq_query(q, k, lam)
    o, _ = oracle.forward(qc, k, v, None, np.zeros((1, 6, 1)), 1e-6, S0)
    for t in range(6):
        np.testing.assert_allclose(o[0, t, 0], S0[0, 0].T @ qc[0, t, 0], rtol=1e-12, atol=1e-13)


def test_a_ccq_mistake_is_caught(tmp_path):
    """Planted in a copy: the sample-covariance divisor n - 1 instead of n."""
    import ctypes
    import subprocess
    src = open(oracle._SRC_CCQ).read()
    bad = src.replace("acc += (M[(size_t)i * dk + j] / n) * qt[j];",
                      "acc += (M[(size_t)i * dk + j] / (n > 1.0 ? n - 1.0 : n)) * qt[j];")
    assert bad != src
    c = tmp_path / "bad_ccq.c"; so = tmp_path / "bad_ccq.so"
    c.write_text(bad)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c)], check=True)
    lib = ctypes.CDLL(str(so))
    dp = ctypes.POINTER(ctypes.c_double)
    lib.ccq_oracle_query.argtypes = [ctypes.c_int] * 4 + [dp] * 10
    q, k, lam = _keys(1)
    qc = np.zeros_like(q)
    p = lambda a: None if a is None else np.ascontiguousarray(a).ctypes.data_as(dp)
    lib.ccq_oracle_query(1, 11, 1, 5, p(q), p(k), p(lam), None, None, None, p(qc), None, None, None)
    K = k[0, :, 0]
    t = 6
    Sig = np.cov(K[:t + 1].T, bias=True)
    assert not np.allclose(qc[0, t, 0], q[0, t, 0] - lam[0, t, 0] * Sig @ q[0, t, 0], rtol=1e-6)
