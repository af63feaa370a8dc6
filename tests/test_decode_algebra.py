"""Two identities the kernels rely on, checked in fp64 against the oracle (no GPU).

* The decode kernel reads the output in the same pass that updates the state: with
  S' = Diag(exp g) S and u = beta (v - S'^T k), o = (S' + k u^T)^T q = S'^T q + (q . k) u, so the
  updated state never has to be read back ("Inside Kimi K3's Architecture", "Kimi Delta
  Attention: the linear core": decay, remove the value the key reads, write, read out).
* The per-token transition is diagonal plus rank one with tied factors,
  (I - beta k k^T) Diag(alpha) = Diag(alpha) - beta k (alpha * k)^T (the "specialised DPLR"
  transition of the same section), which is what lets the chunkwise form use dense tiles.
"""

import numpy as np

import oracle


def test_one_pass_read_out_equals_the_decode_step():
    rng = np.random.default_rng(3)
    N, H, d = 3, 2, 16
    q = rng.standard_normal((N, H, d))
    k = rng.standard_normal((N, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((N, H, d))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((N, H, d))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    S = 0.02 * rng.standard_normal((N, H, d, d))
    o_ref, s_ref = oracle.decode_step(q, k, v, g, beta, S)
    Sd = np.exp(g)[..., None] * S                                   # decay the key rows
    u = beta[..., None] * (v - np.einsum("nhij,nhi->nhj", Sd, k))
    o = np.einsum("nhij,nhi->nhj", Sd, q) + np.einsum("nhi,nhi->nh", q, k)[..., None] * u
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sd + k[..., None] * u[..., None, :], s_ref, rtol=1e-12, atol=1e-12)


def test_transition_is_diagonal_plus_tied_rank_one():
    rng = np.random.default_rng(4)
    d = 7
    k = rng.standard_normal(d)
    k /= np.linalg.norm(k)
    alpha = np.exp(-5.0 / (1.0 + np.exp(-rng.standard_normal(d))))
    beta = 0.7
    lhs = (np.eye(d) - beta * np.outer(k, k)) @ np.diag(alpha)
    rhs = np.diag(alpha) - beta * np.outer(k, alpha * k)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-14, atol=1e-14)
