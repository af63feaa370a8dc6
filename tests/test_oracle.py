"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test names the fact it checks: hand-worked examples (tests/golden), closed forms of
special cases, invariants of the recurrence, and agreement of separately written forms.
A mutation test at the end plants plausible mistakes in a copy of the C source and checks
that the pins here catch every one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def _inputs(B, T, H, dk, dv, seed=0, std=None):
    return ki.prefill_inputs(B, T, H, dk, dv, dtype=torch.float32, seed=seed, state_std=std)


def _args(x):
    return x["q"], x["k"], x["v"], x["g"], x["beta"]


def _rel(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300))


# ----------------------------------------------------------------- hand-worked examples --

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_golden_scalar_hand_example():
    """d_k = d_v = 1: three tokens worked by hand (tests/golden/scalar_dk1_dv1.json)."""
    gd = _golden("scalar_dk1_dv1.json")
    T = len(gd["k"])
    sh = lambda a: torch.tensor(a, dtype=F64).reshape(1, T, 1, 1)
    g = torch.log(torch.tensor(gd["alpha"], dtype=F64)).reshape(1, T, 1, 1)
    beta = torch.tensor(gd["beta"], dtype=F64).reshape(1, T, 1)
    s0 = torch.tensor([[[[gd["s0"]]]]], dtype=F64)
    for fn in (oracle.recurrent, oracle.chunked, oracle.literal):
        kw = dict(chunk=2) if fn is oracle.chunked else {}
        o, s = fn(sh(gd["q"]), sh(gd["k"]), sh(gd["v"]), g, beta, initial_state=s0, **kw)
        np.testing.assert_allclose(o.ravel(), gd["o"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(s.ravel(), [gd["s_final"]], rtol=0, atol=1e-14)


def test_golden_two_channel_hand_example():
    """d_k = d_v = 2: write, per-key-channel decay, delta overwrite, read-back (hand-worked)."""
    gd = _golden("two_channel_overwrite.json")
    T = len(gd["k"])
    t = lambda a: torch.tensor(a, dtype=F64).reshape(1, T, 1, 2)
    g = torch.log(torch.tensor(gd["alpha"], dtype=F64)).reshape(1, T, 1, 2)
    beta = torch.tensor(gd["beta"], dtype=F64).reshape(1, T, 1)
    for fn in (oracle.recurrent, oracle.chunked, oracle.literal):
        kw = dict(chunk=3) if fn is oracle.chunked else {}
        o, s = fn(t(gd["q"]), t(gd["k"]), t(gd["v"]), g, beta, **kw)
        np.testing.assert_allclose(o.reshape(T, 2), gd["o"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(s.reshape(2, 2), gd["S_final"], rtol=0, atol=1e-14)


# -------------------------------------------------------------------- agreement of forms --

@pytest.mark.parametrize("chunk", [1, 3, 16, 64])
def test_chunked_form_equals_recurrence(chunk):
    """Self-check 1: the chunkwise form equals the token recurrence (ragged last chunk,
    random initial state, d_k != d_v)."""
    x = _inputs(2, 77, 3, 16, 12, seed=3, std=0.5)
    o1, s1 = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    o2, s2 = oracle.chunked(*_args(x), initial_state=x["initial_state"], chunk=chunk)
    assert _rel(o2, o1) < 1e-12 and _rel(s2, s1) < 1e-12


def test_chunked_form_full_width_and_saturated_decay():
    """d = 128, chunk 64, with the log-decay at its bound (g = -5 everywhere): the chunkwise
    form needs exp(320) in fp64 and must still agree with the recurrence."""
    x = _inputs(1, 150, 2, 128, 128, seed=4)
    x["g"] = torch.full_like(x["g"], -5.0)
    o1, s1 = oracle.recurrent(*_args(x))
    o2, s2 = oracle.chunked(*_args(x), chunk=64)
    assert _rel(o2, o1) < 1e-10 and _rel(s2, s1) < 1e-10


def test_literal_transition_equals_recurrence():
    """The recurrence with the transition (I - b k k^T) Diag(alpha) formed as a matrix agrees
    with the expanded rank-1 update."""
    x = _inputs(1, 40, 2, 9, 5, seed=5, std=1.0)
    o1, s1 = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    o2, s2 = oracle.literal(*_args(x), initial_state=x["initial_state"])
    assert _rel(o2, o1) < 1e-13 and _rel(s2, s1) < 1e-13


# --------------------------------------------------------------------------- special cases --

def test_beta_zero_from_zero_state_gives_zero():
    """Self-check 2: with beta = 0 nothing is written, so a zero state stays zero and o = 0."""
    x = _inputs(2, 50, 2, 8, 8, seed=6)
    x["beta"] = torch.zeros_like(x["beta"])
    for fn in (oracle.recurrent, oracle.chunked):
        o, s = fn(*_args(x))
        assert np.all(o == 0) and np.all(s == 0)


def test_orthonormal_keys_are_recalled_exactly():
    """Self-check 3: alpha = 1, beta = 1 and orthonormal keys k_1..k_m from a zero state store
    each v_i under k_i; a query q = k_i then returns exactly v_i, and a beta = 0 token leaves
    the state unchanged."""
    dk, dv, m = 16, 10, 12
    rng = np.random.default_rng(7)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :m].T                                   # m orthonormal rows
    vals = rng.standard_normal((m, dv))
    z = lambda *s: torch.zeros(*s, dtype=F64)
    k = torch.tensor(keys).reshape(1, m, 1, dk)
    o, S = oracle.recurrent(k.clone(), k, torch.tensor(vals).reshape(1, m, 1, dv), z(1, m, 1, dk),
                            torch.ones(1, m, 1, dtype=F64))
    for i in range(m):
        qi = torch.tensor(keys[i]).reshape(1, 1, dk)
        oi, S2 = oracle.decode_step(qi, qi, torch.zeros(1, 1, dv, dtype=F64), z(1, 1, dk),
                                    z(1, 1), S)
        np.testing.assert_allclose(oi.ravel(), vals[i], rtol=0, atol=1e-13)
        np.testing.assert_array_equal(S2, S)


def test_decode_continues_prefill():
    """Self-check 4: decode from a T-token prefill's final state equals token T+1 of a
    (T+1)-token prefill, for o and the state."""
    x = _inputs(3, 65, 2, 12, 7, seed=8, std=0.3)
    T = 64
    head = {n: x[n][:, :T] for n in ("q", "k", "v", "g", "beta")}
    o_full, s_full = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    _, s_T = oracle.chunked(*_args(head), initial_state=x["initial_state"], chunk=16)
    last = [x[n][:, T] for n in ("q", "k", "v", "g", "beta")]
    o_dec, s_dec = oracle.decode_step(*last, s_T)
    np.testing.assert_allclose(o_dec, o_full[:, T], rtol=0, atol=1e-12)
    np.testing.assert_allclose(s_dec, s_full, rtol=0, atol=1e-12)


def test_single_token_closed_form():
    """I1: one token from a zero state gives S = beta k v^T and o = beta (q . k) v."""
    x = _inputs(1, 1, 3, 8, 5, seed=9)
    o, S = oracle.recurrent(*_args(x))
    q, k, v, b = (x[n][0, 0].double().numpy() for n in ("q", "k", "v", "beta"))
    for h in range(3):
        np.testing.assert_allclose(S[0, h], b[h] * np.outer(k[h], v[h]), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(o[0, 0, h], b[h] * (q[h] @ k[h]) * v[h], rtol=1e-13, atol=1e-15)


def test_identity_tokens_read_only():
    """I2: g = 0 and beta = 0 leave the state unchanged, and o_t = S_0^T q_t."""
    x = _inputs(2, 20, 2, 8, 6, seed=10, std=1.0)
    x["g"] = torch.zeros_like(x["g"])
    x["beta"] = torch.zeros_like(x["beta"])
    o, S = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    S0 = x["initial_state"].double().numpy()
    np.testing.assert_array_equal(S, S0)
    expect = np.einsum("bthk,bhkv->bthv", x["q"].double().numpy(), S0)
    np.testing.assert_allclose(o, expect, rtol=1e-13, atol=1e-15)


def test_zero_keys_decay_each_channel():
    """I3: with k = 0 only the gate acts: S_t = Diag(exp(sum_{s<=t} g_s)) S_0, so each key
    channel (row) of the state decays on its own, and o_t = S_t^T q_t."""
    x = _inputs(1, 30, 2, 6, 4, seed=11, std=1.0)
    x["k"] = torch.zeros_like(x["k"])
    o, S = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    Gam = np.cumsum(x["g"].double().numpy()[0], axis=0)           # [T, H, dk]
    S0 = x["initial_state"].double().numpy()[0]                    # [H, dk, dv]
    np.testing.assert_allclose(S[0], np.exp(Gam[-1])[..., None] * S0, rtol=1e-13)
    St = np.exp(Gam)[..., None] * S0[None]                          # [T, H, dk, dv]
    expect = np.einsum("thk,thkv->thv", x["q"].double().numpy()[0], St)
    np.testing.assert_allclose(o[0], expect, rtol=1e-12, atol=1e-15)


def test_delta_overwrite():
    """I4: with alpha = 1, beta = 1 and a unit key written twice (v then v'), S^T k = v'
    and the other directions of the state are untouched."""
    dk, dv = 8, 5
    rng = np.random.default_rng(12)
    k = rng.standard_normal(dk); k /= np.linalg.norm(k)
    v1, v2 = rng.standard_normal(dv), rng.standard_normal(dv)
    S0 = rng.standard_normal((dk, dv))
    t = lambda a, d: torch.tensor(np.stack(a)).reshape(1, len(a), 1, d)
    o, S = oracle.recurrent(t([k, k], dk), t([k, k], dk), t([v1, v2], dv),
                            torch.zeros(1, 2, 1, dk, dtype=F64), torch.ones(1, 2, 1, dtype=F64),
                            initial_state=torch.tensor(S0).reshape(1, 1, dk, dv))
    np.testing.assert_allclose(S[0, 0].T @ k, v2, rtol=0, atol=1e-13)
    P = np.eye(dk) - np.outer(k, k)
    np.testing.assert_allclose(P @ S[0, 0], P @ S0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o[0, 1, 0], v2, rtol=0, atol=1e-13)


def test_varlen_equals_separate_runs_and_heads_independent():
    """I5: packed sequences equal separate runs; a head's result ignores the other heads."""
    lengths = [5, 64, 1, 90]
    x = ki.varlen_inputs(lengths, 3, 8, 6, dtype=torch.float32, seed=13, state_std=0.5)
    cu = x["cu_seqlens"].long()
    o, S = oracle.recurrent(*_args(x), cu_seqlens=cu, initial_state=x["initial_state"])
    o2, S2 = oracle.chunked(*_args(x), cu_seqlens=cu, initial_state=x["initial_state"], chunk=16)
    assert _rel(o2, o) < 1e-12 and _rel(S2, S) < 1e-12
    for n in range(len(lengths)):
        a, b = int(cu[n]), int(cu[n + 1])
        part = {m: x[m][:, a:b] for m in ("q", "k", "v", "g", "beta")}
        for h in (0, 2):
            one = {m: part[m][:, :, h:h + 1] for m in part}
            on, Sn = oracle.recurrent(*_args(one), initial_state=x["initial_state"][n:n + 1, h:h + 1])
            np.testing.assert_array_equal(on[0, :, 0], o[0, a:b, h])
            np.testing.assert_array_equal(Sn[0, 0], S[n, h])


def test_state_norm_growth_bound():
    """I6: with unit keys and beta in (0, 1), (I - b k k^T) Diag(alpha) has spectral norm
    <= 1, so ||S_t||_F <= ||S_{t-1}||_F + beta_t ||v_t||."""
    x = _inputs(1, 40, 1, 8, 8, seed=14, std=1.0)
    S = x["initial_state"]
    prev = float(np.linalg.norm(S.double().numpy()))
    for t in range(40):
        step = [x[n][:, t] for n in ("q", "k", "v", "g", "beta")]
        _, S = oracle.decode_step(*step, S)
        cur = float(np.linalg.norm(S))
        b = float(x["beta"][0, t, 0]); vn = float(np.linalg.norm(x["v"][0, t, 0].double().numpy()))
        assert cur <= prev + b * vn + 1e-12
        prev = cur
        S = torch.tensor(S)


@pytest.mark.parametrize("split", [1, 17, 64, 99])
def test_split_prefill_equals_unsplit(split):
    """I8: a prefill split at any token (final state fed back as the initial state) equals
    the unsplit run -- the property a prefill cache relies on."""
    x = _inputs(2, 100, 2, 8, 8, seed=15, std=0.5)
    o, S = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    a = {n: x[n][:, :split] for n in ("q", "k", "v", "g", "beta")}
    b = {n: x[n][:, split:] for n in ("q", "k", "v", "g", "beta")}
    oa, Sa = oracle.chunked(*_args(a), initial_state=x["initial_state"], chunk=16)
    ob, Sb = oracle.chunked(*_args(b), initial_state=torch.tensor(Sa), chunk=16)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Sb, S, rtol=1e-12, atol=1e-14)


def test_scalar_recurrence_random():
    """I9: d_k = d_v = 1 reduces to s_t = (1 - b k^2) a s_{t-1} + b k v, o_t = q s_t,
    evaluated here with plain Python floats."""
    x = _inputs(1, 25, 1, 1, 1, seed=16, std=1.0)
    x["k"] = torch.randn(1, 25, 1, 1, dtype=torch.float32, generator=torch.Generator().manual_seed(1))
    o, S = oracle.recurrent(*_args(x), initial_state=x["initial_state"])
    s = float(x["initial_state"].double().item())
    for t in range(25):
        q, k, v, g = (float(x[n][0, t, 0, 0].double()) for n in ("q", "k", "v", "g"))
        b = float(x["beta"][0, t, 0].double())
        s = (1.0 - b * k * k) * math.exp(g) * s + b * k * v
        assert abs(o[0, t, 0, 0] - q * s) <= 1e-13 * max(1.0, abs(q * s))
    assert abs(S.item() - s) <= 1e-13 * max(1.0, abs(s))


def test_bad_arguments_are_rejected():
    x = _inputs(1, 8, 1, 4, 4, seed=17)
    with pytest.raises(ValueError):
        oracle.recurrent(*_args(x), cu_seqlens=[0, 9])
    with pytest.raises(ValueError):
        oracle.recurrent(*_args(x), initial_state=torch.zeros(2, 1, 4, 4))


# ---------------------------------------------------------------- q/k L2 normalisation -----
# y = x / sqrt(sum x^2 + eps) per row. Pinned by Pythagorean rows (exact unit vectors with
# rational entries), the closed form for a one-hot row, and invariants of a norm.

def test_l2_pythagorean_rows():
    x = np.array([[3.0, 4.0, 0.0], [1.0, 2.0, 2.0], [2.0, -3.0, 6.0], [0.0, 0.0, -5.0]])
    y = oracle.l2_normalize(x, eps=0.0)
    np.testing.assert_allclose(y, [[0.6, 0.8, 0.0], [1 / 3, 2 / 3, 2 / 3], [2 / 7, -3 / 7, 6 / 7], [0.0, 0.0, -1.0]],
                               rtol=0, atol=1e-15)


def test_l2_eps_one_hot_and_zero_rows():
    eps = 1e-6
    x = np.zeros((3, 128))
    x[0, 17] = 1.0
    x[1, 5] = -2.0
    y = oracle.l2_normalize(x, eps=eps)
    assert y[0, 17] == pytest.approx(1.0 / math.sqrt(1.0 + eps), rel=1e-15)
    assert y[1, 5] == pytest.approx(-2.0 / math.sqrt(4.0 + eps), rel=1e-15)
    assert np.count_nonzero(y[:2]) == 2 and np.all(y[2] == 0.0)  # zero row stays zero


def test_l2_invariants():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 4, 64))
    y = oracle.l2_normalize(x, eps=0.0)
    np.testing.assert_allclose((y * y).sum(-1), 1.0, rtol=0, atol=1e-14)           # unit rows
    np.testing.assert_allclose(oracle.l2_normalize(3.5 * x, eps=0.0), y, rtol=0, atol=1e-15)  # scale-free
    np.testing.assert_allclose(oracle.l2_normalize(-x, eps=0.0), -y, rtol=0, atol=0)
    cos = (y * x).sum(-1) / np.sqrt((x * x).sum(-1))                                  # same direction
    np.testing.assert_allclose(cos, 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(oracle.l2_normalize(x[2, 1], eps=0.0), y[2, 1], rtol=0, atol=0)  # rows independent
    ye = oracle.l2_normalize(x, eps=1e-6)                                             # eps shrinks the norm
    ss = (x * x).sum(-1)
    np.testing.assert_allclose((ye * ye).sum(-1), ss / (ss + 1e-6), rtol=1e-13, atol=0)


def test_l2_rejects_bad_eps():
    with pytest.raises(ValueError):
        oracle.l2_normalize(np.ones((2, 3)), eps=-1.0)


# ---------------------------------------------------------------- output gate --------------
# y = o * sigmoid(z). Pinned by closed forms of the logistic function at 0 and +-log(3), its
# limits, and linearity in o.

def test_output_gate_closed_forms():
    o = np.array([2.0, -4.0, 8.0, 1.5, -3.0, 7.0])
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 60.0, -60.0, math.log(7.0)])
    y = oracle.output_gate(o, z)
    np.testing.assert_allclose(y[:3], [1.0, -3.0, 2.0], rtol=0, atol=1e-15)
    assert y[3] == pytest.approx(1.5, rel=1e-15) and abs(y[4]) < 1e-25
    assert y[5] == pytest.approx(7.0 * 7.0 / 8.0, rel=1e-15)


def test_output_gate_linear_in_o_and_symmetric():
    rng = np.random.default_rng(3)
    o, o2, z = rng.standard_normal((3, 4, 5, 16))
    y = oracle.output_gate(o, z)
    np.testing.assert_allclose(oracle.output_gate(o + 2.5 * o2, z), y + 2.5 * oracle.output_gate(o2, z),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(y + oracle.output_gate(o, -z), o, rtol=0, atol=1e-14)  # s(z) + s(-z) = 1


def test_output_gate_rejects_shape_mismatch():
    with pytest.raises(ValueError):
        oracle.output_gate(np.zeros((2, 3)), np.zeros((3, 2)))


# -------------------------------------------------------------- planted-mistake detection --

_PINS = [
    test_golden_scalar_hand_example,
    test_golden_two_channel_hand_example,
    test_beta_zero_from_zero_state_gives_zero,
    test_orthonormal_keys_are_recalled_exactly,
    test_single_token_closed_form,
    test_identity_tokens_read_only,
    test_zero_keys_decay_each_channel,
    test_delta_overwrite,
    test_scalar_recurrence_random,
]

# Plausible mistakes in the recurrence: (description, exact source text, replacement).
_MUTANTS = [
    ("decay the value axis instead of the key axis",
     "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;",
     "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= exp(g[j < dk ? j : 0]);"),
    ("no decay", "double a = exp(g[i]);", "double a = 1.0;"),
    ("decay with exp(-g)", "double a = exp(g[i]);", "double a = exp(-g[i]);"),
    ("wrong sign of the delta correction", "u[j] = beta * (v[j] - kv);", "u[j] = beta * (v[j] + kv);"),
    ("dropped beta", "u[j] = beta * (v[j] - kv);", "u[j] = (v[j] - kv);"),
    ("dropped stale-value term", "u[j] = beta * (v[j] - kv);", "u[j] = beta * v[j];"),
    ("write with q instead of k", "S[(size_t)i * dv + j] += k[i] * u[j];",
     "S[(size_t)i * dv + j] += q[i] * u[j];"),
    ("read out with k instead of q", "acc += S[(size_t)i * dv + j] * q[i];",
     "acc += S[(size_t)i * dv + j] * k[i];"),
    ("transposed state in the correction", "kv += S[(size_t)i * dv + j] * k[i];",
     "kv += S[(size_t)(j < dk ? j : 0) * dv + (i < dv ? i : 0)] * k[j < dk ? j : 0];"),
    ("read-out before the write",
     "    for (int i = 0; i < dk; ++i)\n        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * u[j];\n    /* o_t = S_t^T q_t */",
     "    /* o_t = S_t^T q_t */"),
]


_GATE_PINS = [test_output_gate_closed_forms, test_output_gate_linear_in_o_and_symmetric]
_GATE_MUTANTS = [
    ("sigmoid of -z", "y[i] = o[i] / (1.0 + exp(-z[i]));", "y[i] = o[i] / (1.0 + exp(z[i]));"),
    ("gate added instead of multiplied", "y[i] = o[i] / (1.0 + exp(-z[i]));", "y[i] = o[i] + 1.0 / (1.0 + exp(-z[i]));"),
    ("z as the gate", "y[i] = o[i] / (1.0 + exp(-z[i]));", "y[i] = o[i] * z[i];"),
    ("exp(-z) without the 1", "y[i] = o[i] / (1.0 + exp(-z[i]));", "y[i] = o[i] / exp(-z[i]);"),
]


@pytest.mark.parametrize("idx", range(len(_GATE_MUTANTS)))
def test_output_gate_pins_catch_planted_mistakes(tmp_path, idx):
    desc, old, new = _GATE_MUTANTS[idx]
    text = open(oracle._SRC).read()
    assert text.count(old) == 1, f"mutation site not found: {desc}"
    path = _build_mutant(tmp_path, text.replace(old, new, 1), 200 + idx)
    caught = []
    with oracle.use_library(path):
        for pin in _GATE_PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {desc}"


_L2_PINS = [test_l2_pythagorean_rows, test_l2_eps_one_hot_and_zero_rows, test_l2_invariants]
_L2_MUTANTS = [
    ("no square root", "const double norm = sqrt(ss + eps);", "const double norm = ss + eps;"),
    ("eps outside the root", "const double norm = sqrt(ss + eps);", "const double norm = sqrt(ss) + eps;"),
    ("sum of |x| instead of squares", "ss += x[r * d + i] * x[r * d + i];", "ss += fabs(x[r * d + i]);"),
    ("row stride off by one", "ss += x[r * d + i] * x[r * d + i];", "ss += x[r * (d - 1) + i] * x[r * (d - 1) + i];"),
    ("multiply by the norm", "y[r * d + i] = norm > 0.0 ? x[r * d + i] / norm : 0.0;",
     "y[r * d + i] = x[r * d + i] * norm;"),
]


@pytest.mark.parametrize("idx", range(len(_L2_MUTANTS)))
def test_l2_pins_catch_planted_mistakes(tmp_path, idx):
    desc, old, new = _L2_MUTANTS[idx]
    text = open(oracle._SRC).read()
    assert text.count(old) == 1, f"mutation site not found: {desc}"
    path = _build_mutant(tmp_path, text.replace(old, new, 1), 100 + idx)
    caught = []
    with oracle.use_library(path):
        for pin in _L2_PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {desc}"


def _build_mutant(tmp_path, src_text, i):
    src = tmp_path / f"mutant{i}.c"
    src.write_text(src_text)
    return oracle.build(force=True, src=str(src), out=str(tmp_path / f"libmutant{i}.so"))


@pytest.mark.parametrize("idx", range(len(_MUTANTS)))
def test_pins_catch_planted_mistakes(tmp_path, idx):
    """Each planted mistake in a copy of the C recurrence must fail at least one pin above.
    The mutated copy is built next to the test; the oracle itself is not touched."""
    desc, old, new = _MUTANTS[idx]
    text = open(oracle._SRC).read()
    assert text.count(old) >= 1, f"mutation site not found: {desc}"
    mutated = text.replace(old, new, 1)
    if desc == "read-out before the write":
        # move the write after the read-out loop
        mutated = mutated.replace(
            "        o[j] = acc;\n    }\n}",
            "        o[j] = acc;\n    }\n    for (int i = 0; i < dk; ++i)\n"
            "        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * u[j];\n}", 1)
    path = _build_mutant(tmp_path, mutated, idx)
    caught = []
    with oracle.use_library(path):
        for pin in _PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {desc}"


# ---------------------------------------------------------------- gate from logits -------
# g = -A sigmoid(x): the scaled sigmoid that bounds the log-decay ("Kimi K3 Explained",
# researchpapers.dev, "Architecture at a glance"). Pinned by closed forms of the logistic
# function, not by re-evaluating it.

def test_gate_closed_forms():
    A = 5.0
    x = np.array([0.0, math.log(3.0), -math.log(3.0), math.log(7.0)])
    g = oracle.scaled_sigmoid_gate(x, A)
    np.testing.assert_allclose(g, [-A / 2, -A * 3 / 4, -A / 4, -A * 7 / 8], rtol=0, atol=1e-15)


def test_gate_symmetry_slope_and_range():
    A = 3.25
    x = np.linspace(-30.0, 30.0, 601)
    g = oracle.scaled_sigmoid_gate(x, A)
    gm = oracle.scaled_sigmoid_gate(-x, A)
    np.testing.assert_allclose(g + gm, -A, rtol=0, atol=1e-14)        # sigma(x) + sigma(-x) = 1
    assert np.all(np.diff(g) < 0) and np.all(g < 0) and np.all(g > -A)  # decreasing, in (-A, 0)
    h = 1e-6                                                            # slope at 0 is -A / 4
    slope = (oracle.scaled_sigmoid_gate(np.array([h]), A)[0] - oracle.scaled_sigmoid_gate(np.array([-h]), A)[0]) / (2 * h)
    assert abs(slope + A / 4) < 1e-8
    np.testing.assert_allclose(oracle.scaled_sigmoid_gate(np.array([-50.0, 50.0]), A), [-A * math.exp(-50.0), -A],
                               rtol=1e-12, atol=0)


def test_gate_rejects_bad_bound():
    with pytest.raises(ValueError):
        oracle.scaled_sigmoid_gate(np.zeros(3), 0.0)


# ---------------------------------------------------------------- backward pass -------------
# Gradients of L = sum(do * o) + sum(dS * S_final). Pinned by central finite differences of the
# forward oracle (itself pinned above) and by the closed form of a single token from a zero state.

def _bwd_case(seed=11, dk=3, dv=2, lengths=(4, 3), H=2):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    x = dict(q=rng.standard_normal((1, T, H, dk)), k=rng.standard_normal((1, T, H, dk)) * 0.6,
             v=rng.standard_normal((1, T, H, dv)), g=-rng.uniform(0.05, 1.5, (1, T, H, dk)),
             beta=rng.uniform(0.2, 0.9, (1, T, H)))
    N = len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    init = rng.standard_normal((N, H, dk, dv)) * 0.5
    do = rng.standard_normal((1, T, H, dv))
    dfin = rng.standard_normal((N, H, dk, dv))
    return x, cu, init, do, dfin


def _loss(x, cu, init, do, dfin):
    o, fin = oracle.recurrent(*(x[n] for n in ("q", "k", "v", "g", "beta")), cu_seqlens=cu, initial_state=init)
    return float((o * do).sum() + (fin * dfin).sum())


def test_backward_matches_central_differences():
    x, cu, init, do, dfin = _bwd_case()
    grads = oracle.backward(*(x[n] for n in ("q", "k", "v", "g", "beta")), do, dfin, cu_seqlens=cu,
                            initial_state=init)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), (None, "d_initial_state")):
        base = init if name is None else x[name]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            saved = base[idx]
            base[idx] = saved + h
            lp = _loss(x, cu, init, do, dfin)
            base[idx] = saved - h
            lm = _loss(x, cu, init, do, dfin)
            base[idx] = saved
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grads[gname], fd, rtol=1e-6, atol=1e-7, err_msg=gname)


def test_backward_single_token_closed_form():
    # From a zero state one token gives S = beta k v^T and o = beta (q.k) v, so with dS_final = 0:
    # dq = beta (v.do) k, dk = beta (v.do) q, dv = beta (q.k) do, dbeta = (q.k)(v.do), dg = 0 (it
    # multiplies the zero state), and, since S1 = (I - beta k k^T) Diag(alpha) S0 + beta k v^T,
    # dS0 = Diag(alpha) (q - beta (k.q) k) do^T.
    rng = np.random.default_rng(5)
    q, k, v, do = rng.standard_normal(4), rng.standard_normal(4), rng.standard_normal(3), rng.standard_normal(3)
    b = 0.7
    r = lambda a: a.reshape(1, 1, 1, -1)
    grads = oracle.backward(r(q), r(k), r(v), r(-np.full(4, 0.3)), np.full((1, 1, 1), b), r(do))
    qk, vdo = q @ k, v @ do
    np.testing.assert_allclose(grads["dq"].ravel(), b * vdo * k, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(grads["dk"].ravel(), b * vdo * q, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(grads["dv"].ravel(), b * qk * do, rtol=1e-13, atol=1e-14)
    assert grads["dbeta"].item() == pytest.approx(qk * vdo, rel=1e-13)
    assert np.all(grads["dg"] == 0.0)
    ds0 = np.outer(np.exp(-0.3) * (q - b * qk * k), do)
    np.testing.assert_allclose(grads["d_initial_state"].reshape(4, 3), ds0, rtol=1e-13, atol=1e-14)


_BWD_PINS = [test_backward_matches_central_differences, test_backward_single_token_closed_form]
_BWD_MUTANTS = [
    ("state gradient not decayed", "dS[(size_t)i * dv + j] = a * dSd[(size_t)i * dv + j];",
     "dS[(size_t)i * dv + j] = dSd[(size_t)i * dv + j];"),
    ("dropped k-read term of dSd", "dSd[(size_t)i * dv + j] = dS[(size_t)i * dv + j] - kt[i] * bt * du[j];",
     "dSd[(size_t)i * dv + j] = dS[(size_t)i * dv + j];"),
    ("wrong sign in dk", "acc += dS[(size_t)i * dv + j] * bt * w[j] - Sd[(size_t)i * dv + j] * bt * du[j];",
     "acc += dS[(size_t)i * dv + j] * bt * w[j] + Sd[(size_t)i * dv + j] * bt * du[j];"),
    ("dv without beta", "dvv[r * dv + j] = bt * du[j];", "dvv[r * dv + j] = du[j];"),
    ("read-out gradient from the pre-write state", "acc += St[(size_t)i * dv + j] * dot[j];",
     "acc += Sd[(size_t)i * dv + j] * dot[j];"),
    ("dg against the undecayed state", "acc += dSd[(size_t)i * dv + j] * Sd[(size_t)i * dv + j];",
     "acc += dSd[(size_t)i * dv + j] * Sp[(size_t)i * dv + j];"),
]


@pytest.mark.parametrize("idx", range(len(_BWD_MUTANTS)))
def test_backward_pins_catch_planted_mistakes(tmp_path, idx):
    desc, old, new = _BWD_MUTANTS[idx]
    text = open(oracle._SRC).read()
    assert text.count(old) == 1, f"mutation site not found: {desc}"
    path = _build_mutant(tmp_path, text.replace(old, new, 1), 300 + idx)
    caught = []
    with oracle.use_library(path):
        for pin in _BWD_PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {desc}"
