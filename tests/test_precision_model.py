"""The kernels' precision schemes, emulated in numpy and held to the parity bar (no GPU).

Each emulation restates, at the level of rounding, what a kernel computes; it shares no code with
the CUDA path and is compared with the fp64 oracle on the workloads' inputs and on the method's
degenerate inputs (no decay, g = -5 everywhere, beta = 0, k = 0):

* the tensor-core prefill: bf16 MMA operands (the decay-scaled K and Q tiles of A and P with their
  per-half reference rows, the bf16 state copy, -K+ S, T, U, P, Khat), fp32 accumulation and
  state, the 16 x 16 diagonal blocks of the inverse in fp32 and its 16 -> 32 -> 64 merges in tf32,
  o rounded to bf16 once;
* the d = 128 backward for bf16 inputs: tf32 rounding of the operands of the products with the
  128 x 128 states and of P^T dO, fp32-accurate (3 x tf32) products elsewhere.
* the split along the sequence: the local pass and the transition pass (v = 0 from the identity)
  as tensor-core prefills, the scan S_start <- M S_start + S_loc in fp32, and the correction
  o += q~ S_start from bf16 q~ and S_start onto the already rounded o, rounded again.

On GB300 the emulations reproduce the measured errors of the existing cases within about 1.5x, so
a change of either scheme can be checked against the bar here before it reaches a GPU.
"""

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle

NAMES = ("q", "k", "v", "g", "beta")
MAX_ABS, REL_FROB = 2e-2, 5e-3


def bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def tf32(x):
    """Round to tf32 (10 mantissa bits, nearest with ties away from zero)."""
    a = np.asarray(x, dtype=np.float32)
    u = (a.view(np.uint32).copy() + np.uint32(0x1000)) & np.uint32(0xFFFFE000)
    return u.view(np.float32).astype(np.float64)


def f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def degenerate(x, kind):
    if kind == "no_decay":
        x["g"] = torch.zeros_like(x["g"])
    elif kind == "saturated":
        x["g"] = torch.full_like(x["g"], -5.0)
    elif kind == "beta0":
        x["beta"] = torch.zeros_like(x["beta"])
        x["g"] = x["g"] * 0.1
    elif kind == "k0":
        x["k"] = torch.zeros_like(x["k"])
        x["g"] = x["g"] * 0.1
    return x


# ----------------------------------------------------------------------- tensor-core prefill ---

def _prefill_inverse(A):
    X = np.zeros((64, 64))
    for o in range(0, 64, 16):
        X[o:o + 16, o:o + 16] = f32(np.linalg.inv(np.eye(16) + A[o:o + 16, o:o + 16]))
    for half in (16, 32):
        for lo in range(0, 64, 2 * half):
            a, b = slice(lo, lo + half), slice(lo + half, lo + 2 * half)
            Y = f32(tf32(A[b, a]) @ tf32(X[a, a]))
            X[b, a] = -f32(tf32(X[b, b]) @ tf32(Y))
    return X


def _prefill_chunk(S, q, k, v, g, beta):
    L = q.shape[0]
    if L < 64:  # rows past the end act as identity tokens (zero inputs)
        z = lambda t: np.vstack([t, np.zeros((64 - L,) + t.shape[1:])])
        q, k, v, g, beta = z(q), z(k), z(v), z(g), np.concatenate([beta, np.zeros(64 - L)])
    G = f32(np.cumsum(g, 0))
    A = np.zeros((64, 64))
    P = np.zeros((64, 64))
    for lo, ref in ((0, G[15]), (32, G[47])):
        r = slice(lo, lo + 32)
        f, fi = np.exp(np.clip(G[r] - ref, -87, 87)), np.exp(np.clip(ref - G[r], -87, 87))
        with np.errstate(over="ignore", invalid="ignore"):
            A[r, r] = f32(bf16(k[r] * f) @ bf16(k[r] * fi).T)
            P[r, r] = f32(bf16(q[r] * f) @ bf16(k[r] * fi).T)
    rb, ca = slice(32, 64), slice(0, 32)
    er, ec = np.exp(G[rb] - G[31]), np.exp(G[31] - G[ca])
    A[rb, ca] = f32(bf16(k[rb] * er) @ bf16(k[ca] * ec).T)
    P[rb, ca] = f32(bf16(q[rb] * er) @ bf16(k[ca] * ec).T)
    A = np.where(np.tril(np.ones((64, 64), bool), -1), f32(A * beta[:, None]), 0.0)  # selected, not multiplied
    P = bf16(np.where(np.tril(np.ones((64, 64), bool)), P, 0.0))
    T = bf16(_prefill_inverse(A) * beta[None, :])
    gam = np.exp(G)
    kp, qp, kh = bf16(k * gam), bf16(q * gam), bf16(k * np.exp(G[63] - G))
    Sb = bf16(S)
    KS, QS = f32(kp @ Sb), f32(qp @ Sb)
    U = bf16(f32(T @ bf16(v) + T @ bf16(-KS)))
    O = bf16(f32(QS + P @ U))
    return f32(f32(S * gam[63][:, None]) + f32(kh.T @ U)), O[:L]


def prefill_model(q, k, v, g, beta, S0):
    S, o = S0.copy(), np.zeros_like(v)
    for t0 in range(0, q.shape[0], 64):
        sl = slice(t0, min(t0 + 64, q.shape[0]))
        S, o[sl] = _prefill_chunk(S, q[sl], k[sl], v[sl], g[sl], beta[sl])
    return o, S


def split_model(q, k, v, g, beta, S0, P):
    """The split path with P segments of a multiple of 64 rows."""
    T = q.shape[0]
    per = -(-T // P)              # ceil(T / P)
    Ls = -(-per // 64) * 64       # rounded up to whole chunks
    o, S_start = np.zeros_like(v), S0.copy()
    for t0 in range(0, T, Ls):
        sl = slice(t0, min(t0 + Ls, T))
        o_loc, s_loc = prefill_model(q[sl], k[sl], v[sl], g[sl], beta[sl], np.zeros_like(S0))
        qt, M = prefill_model(q[sl], k[sl], np.zeros_like(v[sl]), g[sl], beta[sl], np.eye(S0.shape[0]))
        o[sl] = bf16(f32(o_loc + f32(qt @ bf16(S_start))))
        S_start = f32(f32(M @ S_start) + s_loc)
    return o, S_start


# ---------------------------------------------------------------- d = 128 backward, bf16 inputs ---

def _bwd_forward(S, q, k, v, g, beta):
    gam = np.exp(np.cumsum(g, 0))
    gC = gam[-1]
    Kp, Km, Qp, Kc = k * gam, k / gam, q * gam, k * gC / gam
    Ab = Kp @ Km.T
    X = np.linalg.inv(np.eye(len(beta)) + np.tril(beta[:, None] * Ab, -1))
    T = X * beta[None, :]
    R = v - tf32(Kp) @ tf32(S)
    U = T @ R
    P = np.tril(Qp @ Km.T)
    S_next = gC[:, None] * S + tf32(Kc).T @ tf32(U)
    return S_next, dict(gam=gam, gC=gC, Kp=Kp, Km=Km, Qp=Qp, Kc=Kc, Ab=Ab, X=X, T=T, R=R, U=U, P=P)


def _bwd_adjoint(S, dO, dSn, beta, f):
    gam, gC, Kp, Km, Qp, Kc = (f[n] for n in ("gam", "gC", "Kp", "Km", "Qp", "Kc"))
    Ab, X, T, R, U, P = (f[n] for n in ("Ab", "X", "T", "R", "U", "P"))
    dU = tf32(P).T @ tf32(dO) + tf32(Kc) @ tf32(dSn)
    dR = T.T @ dU
    dP = np.tril(dO @ U.T)
    dT = dU @ R.T
    dA = np.tril(-X.T @ (dT * beta[None, :]) @ X.T, -1)
    dbeta = np.sum(X * dT, 0) + np.sum(dA * Ab, 1)
    dAb = beta[:, None] * dA
    dQp = tf32(dO) @ tf32(S).T + dP @ Km
    dKp = -(tf32(dR) @ tf32(S).T) + dAb @ Km
    dKm = dP.T @ Qp + dAb.T @ Kp
    dKc = tf32(U) @ tf32(dSn).T
    dk = dKp * gam + dKm / gam + dKc * gC / gam
    dGam = dKp * Kp - dKm * Km + dQp * Qp - dKc * Kc
    dGam[-1] += np.sum(dKc * Kc, 0) + np.sum(dSn * S, 1) * gC
    dS = tf32(Qp).T @ tf32(dO) - tf32(Kp).T @ tf32(dR) + gC[:, None] * dSn
    return dQp * gam, dk, dR, np.cumsum(dGam[::-1], 0)[::-1], dbeta, dS


def backward_model(q, k, v, g, beta, dO, S0, C=16):
    starts = list(range(0, q.shape[0], C))
    states, S = [], S0.copy()
    for t0 in starts:
        sl = slice(t0, min(t0 + C, q.shape[0]))
        states.append(S)
        S, _ = _bwd_forward(S, q[sl], k[sl], v[sl], g[sl], beta[sl])
    out = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    dS = np.zeros_like(S0)
    for t0, S in zip(reversed(starts), reversed(states)):
        sl = slice(t0, min(t0 + C, q.shape[0]))
        _, f = _bwd_forward(S, q[sl], k[sl], v[sl], g[sl], beta[sl])
        grads = _bwd_adjoint(S, dO[sl], dS, beta[sl], f)
        for n, val in zip(("dq", "dk", "dv", "dg", "dbeta"), grads[:5]):
            out[n][sl] = val
        dS = grads[5]
    out["d_initial_state"] = dS
    return out


# ------------------------------------------------------------------------------------ tests ---

def _check(got, ref, name):
    err = np.abs(got - ref).max(initial=0.0)
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nr if nr > 1e-30 else 0.0
    assert err <= MAX_ABS and rel <= REL_FROB, f"{name}: max-abs {err:.2e}, rel-Frob {rel:.2e}"
    return rel


@pytest.mark.parametrize("kind", ["workload", "no_decay", "saturated", "beta0", "k0"])
def test_prefill_precision_scheme_meets_the_bar(kind):
    x = degenerate(ki.prefill_inputs(1, 150, 2, 128, 128, seed=41, state_std=0.02), kind)
    ro, rs = oracle.recurrent(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    for h in range(2):
        a = lambda t: t[0, :, h].double().numpy()
        o, S = prefill_model(a(x["q"]), a(x["k"]), a(x["v"]), a(x["g"]), x["beta"][0, :, h].double().numpy(),
                             x["initial_state"][0, h].double().numpy())
        rel = _check(o, ro[0, :, h], f"o ({kind}, h={h})")
        assert rel > 1e-4, "the emulation must carry the bf16 rounding (a vanishing error means it does not)"
        _check(S, rs[0, h], f"final state ({kind}, h={h})")


@pytest.mark.parametrize("kind", ["workload", "no_decay", "saturated", "beta0", "k0"])
def test_backward_precision_scheme_meets_the_bar(kind):
    x = degenerate(ki.prefill_inputs(1, 70, 1, 128, 128, seed=43, state_std=0.02), kind)
    do = ki.gate_logits_like(x["v"], seed=44)
    ref = oracle.backward(*(x[n] for n in NAMES), do, initial_state=x["initial_state"])
    a = lambda t: t[0, :, 0].double().numpy()
    got = backward_model(a(x["q"]), a(x["k"]), a(x["v"]), a(x["g"]), x["beta"][0, :, 0].double().numpy(), a(do),
                         x["initial_state"][0, 0].double().numpy())
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        _check(got[n], ref[n][0, :, 0], f"{n} ({kind})")
    _check(got["d_initial_state"], ref["d_initial_state"][0, 0], f"d_initial_state ({kind})")


@pytest.mark.parametrize("decay", [1.0, 0.002])
def test_split_precision_scheme_meets_the_bar(decay):
    """8192 tokens in 4 segments, with the workloads' gates and with log-decays in (-0.01, 0) (each
    segment's start state matters for its whole length)."""
    x = ki.prefill_inputs(1, 8192, 1, 128, 128, seed=52, state_std=0.02)
    x["g"] = (x["g"].float() * decay).to(torch.bfloat16)
    ro, rs = oracle.recurrent(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    a = lambda t: t[0, :, 0].double().numpy()
    o, S = split_model(a(x["q"]), a(x["k"]), a(x["v"]), a(x["g"]), x["beta"][0, :, 0].double().numpy(),
                       x["initial_state"][0, 0].double().numpy(), 4)
    _check(o, ro[0, :, 0], f"o (decay x{decay})")
    _check(S, rs[0, 0], f"final state (decay x{decay})")
