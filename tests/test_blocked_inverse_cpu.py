"""The blocked inverse of the UT/WY solve equals the plain inverse.

Phase 1 forms T = (I + L)^{-1} for the strictly lower 64 x 64 matrix
L = strict_lower(diag(beta) (Gamma o K K^T)) of a chunk (the block solver of
Gated DeltaNet with B = Diag(beta), Kaczmarz Linear Attention summary,
gist.science 2605.08587, "Implementacao") in three levels: the four 16 x 16
diagonal blocks by forward substitution, then twice
[[A, 0], [C, B]]^{-1} = [[D1, 0], [X, D2]] with D1 = A^{-1}, D2 = B^{-1} and
X = -D2 C D1 (block sizes 16 -> 32 -> 64).  This file restates those steps in
numpy fp64 (test only) and checks them against numpy's inverse, for the
chunk's matrix as the kernels see it (including a ragged chunk, whose rows
past its end are zero).
"""
import numpy as np
import pytest


def forward_substitution_inverse(A):
    """Inverse of a unit lower-triangular matrix, one column at a time."""
    n = A.shape[0]
    X = np.zeros_like(A)
    for c in range(n):
        for r in range(n):
            X[r, c] = (1.0 if r == c else 0.0) - A[r, :r] @ X[:r, c]
    return X


def blocked_inverse(L):
    n = L.shape[0]
    T = np.eye(n) + L
    for o in range(0, n, 16):
        T[o:o + 16, o:o + 16] = forward_substitution_inverse(np.eye(16) + L[o:o + 16, o:o + 16])
    for size in (16, 32):
        for o in range(0, n, 2 * size):
            D1 = T[o:o + size, o:o + size]
            D2 = T[o + size:o + 2 * size, o + size:o + 2 * size]
            C = T[o + size:o + 2 * size, o:o + size]
            T[o + size:o + 2 * size, o:o + size] = -D2 @ C @ D1
    return T


def _chunk_L(seed, nc):
    """L of one chunk: beta, the decay matrix and the keys drawn like the
    workloads (nc live rows; rows and columns past nc are zero)."""
    rng = np.random.default_rng(seed)
    d = 128
    k = rng.standard_normal((64, d)) / np.sqrt(d) * np.exp(0.5 * rng.standard_normal((64, 1)))
    eta = 1.0 / (1.0 + np.exp(-rng.standard_normal(64)))
    beta = eta / (np.sum(k * k, axis=1) + 1e-6)
    g = np.cumsum(-np.log1p(np.exp(rng.standard_normal(64))))
    Gam = np.exp(np.minimum(g[:, None] - g[None, :], 0.0))
    L = np.tril(beta[:, None] * Gam * (k @ k.T), -1)
    L[nc:, :] = 0.0
    L[:, nc:] = 0.0
    return L


@pytest.mark.parametrize("seed,nc", [(0, 64), (1, 64), (2, 37), (3, 1)])
def test_blocked_inverse_equals_inverse(seed, nc):
    L = _chunk_L(seed, nc)
    ref = np.linalg.inv(np.eye(64) + L)
    got = blocked_inverse(L)
    assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())
    # the inverse stays unit lower triangular: the zeros the merges skip are exact
    assert np.array_equal(np.triu(got, 1), np.zeros((64, 64)))
    assert np.array_equal(np.diag(got), np.ones(64))


def test_a_merge_mistake_is_caught():
    """X = -D1 C D2 (factors swapped) must not give the inverse."""
    L = _chunk_L(5, 64)
    T = np.eye(64) + L
    for o in range(0, 64, 16):
        T[o:o + 16, o:o + 16] = forward_substitution_inverse(np.eye(16) + L[o:o + 16, o:o + 16])
    for size in (16, 32):
        for o in range(0, 64, 2 * size):
            D1 = T[o:o + size, o:o + size]
            D2 = T[o + size:o + 2 * size, o + size:o + 2 * size]
            C = T[o + size:o + 2 * size, o:o + size]
            T[o + size:o + 2 * size, o:o + size] = -D1 @ C @ D2
    ref = np.linalg.inv(np.eye(64) + L)
    assert np.abs(T - ref).max() > 1e-6 * np.abs(ref).max()
