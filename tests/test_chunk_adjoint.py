"""The chunkwise adjoint that the d = 128 backward kernel evaluates, restated here in fp64 numpy
and checked against the oracle's token-by-token adjoint (itself pinned by finite differences).

This pins the algebra of the kernel's derivation, not the kernel: the pages train the model
("Kimi K3 Explained", researchpapers.dev, "Architecture at a glance") but give no gradient method,
so the chunkwise form of the recurrence ("Inside Kimi K3's Architecture", "Kimi Delta Attention:
the linear core": the chunkwise algorithm on the diagonal-plus-low-rank transition) is
differentiated by hand. Per chunk of C rows, with S the state at its start and
Gam = cumsum(g), gam = exp(Gam), gC = gam of the chunk's last row:

    Kp = K gam, Km = K / gam, Qp = Q gam, Kc = K gC / gam
    Ab = Kp Km^T, A = strict_lower(Diag(beta) Ab), X = (I + A)^-1, T = X Diag(beta)
    R = V - Kp S, U = T R, P = lower(Qp Km^T), O = Qp S + P U, S' = Diag(gC) S + Kc^T U

and, given dO and dS' (the gradient with respect to S'), the adjoint written below.
"""

import numpy as np
import pytest

import oracle


def _chunk_forward(S, q, k, v, g, beta):
    Gam = np.cumsum(g, axis=0)
    gam = np.exp(Gam)
    gC = gam[-1]
    Kp, Km, Qp = k * gam, k / gam, q * gam
    Kc = k * gC / gam
    Ab = Kp @ Km.T
    A = np.tril(beta[:, None] * Ab, -1)
    X = np.linalg.inv(np.eye(len(beta)) + A)
    T = X * beta[None, :]
    R = v - Kp @ S
    U = T @ R
    P = np.tril(Qp @ Km.T)
    O = Qp @ S + P @ U
    S_next = gC[:, None] * S + Kc.T @ U
    return O, S_next, dict(gam=gam, gC=gC, Kp=Kp, Km=Km, Qp=Qp, Kc=Kc, Ab=Ab, X=X, T=T, R=R, U=U, P=P)


def _chunk_adjoint(S, dO, dS_next, beta, f):
    gam, gC, Kp, Km, Qp, Kc = f["gam"], f["gC"], f["Kp"], f["Km"], f["Qp"], f["Kc"]
    Ab, X, T, R, U, P = f["Ab"], f["X"], f["T"], f["R"], f["U"], f["P"]
    dU = P.T @ dO + Kc @ dS_next
    dR = T.T @ dU                                   # = dV
    dP = np.tril(dO @ U.T)
    dT = dU @ R.T
    dX = dT * beta[None, :]
    dA = np.tril(-X.T @ dX @ X.T, -1)
    dbeta = np.sum(X * dT, axis=0) + np.sum(dA * Ab, axis=1)
    dAb = beta[:, None] * dA                        # Diag(beta) dA
    dQp = dO @ S.T + dP @ Km
    dKp = -dR @ S.T + dAb @ Km
    dKm = dP.T @ Qp + dAb.T @ Kp
    dKc = U @ dS_next.T
    dgC = np.sum(dS_next * S, axis=1)
    dk = dKp * gam + dKm / gam + dKc * gC / gam
    dq = dQp * gam
    dGam = dKp * Kp - dKm * Km + dQp * Qp - dKc * Kc
    dGam[-1] += np.sum(dKc * Kc, axis=0) + dgC * gC
    dg = np.cumsum(dGam[::-1], axis=0)[::-1]        # reverse cumsum over the rows
    dS = Qp.T @ dO - Kp.T @ dR + gC[:, None] * dS_next
    return dq, dk, dR, dg, dbeta, dS


def _chunkwise_backward(q, k, v, g, beta, d_o, S0, dS_fin, C):
    """One (sequence, head): forward sweep keeping each chunk's start state, then the reverse."""
    T = q.shape[0]
    starts = list(range(0, T, C))
    states, S = [], S0.copy()
    for t0 in starts:
        sl = slice(t0, min(t0 + C, T))
        states.append(S)
        _, S, _ = _chunk_forward(S, q[sl], k[sl], v[sl], g[sl], beta[sl])
    out = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    dS = dS_fin.copy()
    for t0, S in zip(reversed(starts), reversed(states)):
        sl = slice(t0, min(t0 + C, T))
        _, _, f = _chunk_forward(S, q[sl], k[sl], v[sl], g[sl], beta[sl])
        dq, dk, dv, dg, db, dS = _chunk_adjoint(S, d_o[sl], dS, beta[sl], f)
        out["dq"][sl], out["dk"][sl], out["dv"][sl], out["dg"][sl], out["dbeta"][sl] = dq, dk, dv, dg, db
    out["d_initial_state"] = dS
    return out


@pytest.mark.parametrize("T,C,decay", [(37, 16, 1.0), (16, 16, 1.0), (5, 16, 1.0), (50, 8, 1.0), (37, 16, 0.02),
                                         (16, 16, 0.02)])
def test_chunkwise_adjoint_matches_token_adjoint(T, C, decay):
    """decay scales the log-decays: 1 gives the workloads' gates, 0.02 a slow decay whose state
    and gate terms (S, dS', gC) carry across chunks at full weight."""
    rng = np.random.default_rng(T * 100 + C)
    H, dk, dv = 2, 8, 6
    q = rng.standard_normal((1, T, H, dk))
    k = rng.standard_normal((1, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, H, dv))
    g = -5.0 * decay / (1.0 + np.exp(-rng.standard_normal((1, T, H, dk))))   # log-decays in [-5, 0]
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, H))))
    S0 = 0.1 * rng.standard_normal((1, H, dk, dv))
    d_o = rng.standard_normal((1, T, H, dv))
    dS_fin = rng.standard_normal((1, H, dk, dv))
    ref = oracle.backward(q, k, v, g, beta, d_o, dS_fin, initial_state=S0)
    for h in range(H):
        got = _chunkwise_backward(q[0, :, h], k[0, :, h], v[0, :, h], g[0, :, h], beta[0, :, h], d_o[0, :, h],
                                  S0[0, h], dS_fin[0, h], C)
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            r = ref[name][0, :, h]
            np.testing.assert_allclose(got[name], r, rtol=1e-9, atol=1e-9 * max(1.0, np.abs(r).max()), err_msg=name)
        r = ref["d_initial_state"][0, h]
        np.testing.assert_allclose(got["d_initial_state"], r, rtol=1e-9, atol=1e-9 * max(1.0, np.abs(r).max()))


def test_chunkwise_forward_matches_recurrence():
    """The forward form the adjoint differentiates gives the oracle recurrence's o and final state."""
    rng = np.random.default_rng(7)
    T, H, dk, dv, C = 45, 1, 8, 8, 16
    q = rng.standard_normal((1, T, H, dk))
    k = rng.standard_normal((1, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, H, dv))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((1, T, H, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, H))))
    S0 = 0.1 * rng.standard_normal((1, H, dk, dv))
    o_ref, s_ref = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    S = S0[0, 0].copy()
    for t0 in range(0, T, C):
        sl = slice(t0, min(t0 + C, T))
        O, S, _ = _chunk_forward(S, q[0, sl, 0], k[0, sl, 0], v[0, sl, 0], g[0, sl, 0], beta[0, sl, 0])
        np.testing.assert_allclose(O, o_ref[0, sl, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, s_ref[0, 0], rtol=1e-10, atol=1e-10)
