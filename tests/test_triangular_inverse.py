"""The two triangular solves of the kernels, restated in float32 numpy and held to a dense fp64
inverse (no GPU).

The chunkwise form needs T = (I + A)^{-1} Diag(beta) with A = strict_lower(Diag(beta) K+ K-^T)
("Kimi K3 Explained", researchpapers.dev, "Architecture at a glance": the chunkwise computation
on dense tiles). Both kernels invert the unit lower-triangular I + A by blocks, using that for
I + A = [[I + A11, 0], [A21, I + A22]] the inverse is [[X11, 0], [-X22 A21 X11, X22]]:

* the prefill (64 rows): 4 x 4 diagonal blocks in closed form, then merges 4 -> 8 -> 16 inside
  each 16-row block, then 16 -> 32 and 32 -> 64 across blocks;
* the backward (16 rows): the two 8 x 8 diagonal blocks by forward substitution, one merge.
"""

import numpy as np
import pytest

f32 = np.float32


def _inv4(A):
    """Closed form of (I + A)^{-1} for a 4 x 4 strictly lower A."""
    X = np.eye(4, dtype=f32)
    X[1, 0] = -A[1, 0]
    X[2, 1] = -A[2, 1]
    X[3, 2] = -A[3, 2]
    X[2, 0] = -(A[2, 0] + A[2, 1] * X[1, 0])
    X[3, 1] = -(A[3, 1] + A[3, 2] * X[2, 1])
    X[3, 0] = -(A[3, 0] + A[3, 1] * X[1, 0] + A[3, 2] * X[2, 0])
    return X


def _merge(X, A, lo, half):
    """Fill X21 of the block [lo, lo + 2 half) from its two inverted diagonal halves."""
    a, b = slice(lo, lo + half), slice(lo + half, lo + 2 * half)
    X[b, a] = -(X[b, b] @ (A[b, a] @ X[a, a]))


def prefill_inverse(A):
    n = A.shape[0]
    X = np.zeros((n, n), f32)
    for o in range(0, n, 4):
        X[o:o + 4, o:o + 4] = _inv4(A[o:o + 4, o:o + 4])
    for half in (4, 8, 16, 32):
        for lo in range(0, n, 2 * half):
            _merge(X, A, lo, half)
    return X


def backward_inverse(A):
    X = np.zeros((16, 16), f32)
    for lo in (0, 8):  # forward substitution per column inside the 8 x 8 diagonal block
        for j in range(lo, lo + 8):
            X[j, j] = 1.0
            for i in range(j + 1, lo + 8):
                X[i, j] = -np.dot(A[i, j:i], X[j:i, j])
    _merge(X, A, 0, 8)
    return X


def _workload_A(n, rng, decay=1.0):
    """A = strict_lower(Diag(beta) K+ K-^T) for unit keys, beta = sigmoid(N(0,1)) and log-decays
    -5 sigmoid(N(0,1)) (scaled by `decay`), built in fp64."""
    d = 64
    k = rng.standard_normal((n, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    g = -5.0 * decay / (1.0 + np.exp(-rng.standard_normal((n, d))))
    Gam = np.cumsum(g, axis=0)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(n)))
    Ab = np.einsum("rc,sc,rsc->rs", k, k, np.exp(np.minimum(Gam[:, None, :] - Gam[None, :, :], 0.0)))
    return np.tril(beta[:, None] * Ab, -1)


@pytest.mark.parametrize("decay", [1.0, 0.05, 0.0])
def test_prefill_doubling_inverse(decay):
    rng = np.random.default_rng(int(decay * 100))
    A = _workload_A(64, rng, decay)
    ref = np.linalg.inv(np.eye(64) + A)
    got = prefill_inverse(A.astype(f32)).astype(np.float64)
    assert np.all(np.triu(got, 1) == 0) and np.all(np.diag(got) == 1)
    np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5 * max(1.0, np.abs(ref).max()))


@pytest.mark.parametrize("decay", [1.0, 0.05, 0.0])
def test_backward_blocked_inverse(decay):
    rng = np.random.default_rng(7 + int(decay * 100))
    A = _workload_A(16, rng, decay)
    ref = np.linalg.inv(np.eye(16) + A)
    got = backward_inverse(A.astype(f32)).astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * max(1.0, np.abs(ref).max()))


def test_closed_form_4x4_against_exact_arithmetic():
    """Integer entries: the closed form gives the exact inverse (all values are small integers)."""
    A = np.tril(np.arange(1, 17, dtype=np.float64).reshape(4, 4), -1)
    want = np.linalg.inv(np.eye(4) + A)
    np.testing.assert_array_equal(_inv4(A.astype(f32)).astype(np.float64), np.round(want))
