"""The prefill options and the backward pass at the headline size (B=4, T=8192, H=32, d=128,
bf16; the launch configuration bench.py times), checked on sampled (batch row, head) pairs that
the oracle computes one by one."""

import math

import pytest
import torch

import gated_delta_rule_56_gb300 as kda
import kda_inputs as ki
import oracle
from kda_testutil import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NAMES = ("q", "k", "v", "g", "beta")
B, T, H, D = 4, 8192, 32, 128
PAIRS = [(0, 0), (3, 31), (2, 9)]


@pytest.fixture(scope="module")
def x():
    kda.load()
    return ki.prefill_inputs(B, T, H, D, D, device=DEV, seed=0)


def _pair(t, b, h, rows=None):
    sl = slice(None) if rows is None else slice(*rows)
    return t[b:b + 1, sl, h:h + 1].cpu()


def _unit(t):  # the oracle's fp64 normalisation of the raw rows
    return oracle.l2_normalize(t.cpu())


def test_full_size_gate_logits_l2norm_and_output_gate(x):
    xg = ki.gate_logits_like(x["g"], seed=1)
    q, k = ki.raw_qk_like(x["q"], seed=2), ki.raw_qk_like(x["k"], seed=3)
    z = ki.gate_logits_like(x["v"], seed=4)
    o, s = kda.prefill(q, k, x["v"], xg, x["beta"], gate_bound=5.0, qk_l2norm=True, out_gate=z)
    kda.check_status()
    for b, h in PAIRS:
        g = oracle.scaled_sigmoid_gate(_pair(xg, b, h), 5.0)
        ro, rs = oracle.recurrent(_unit(_pair(q, b, h)), _unit(_pair(k, b, h)), _pair(x["v"], b, h), g,
                                  _pair(x["beta"], b, h))
        assert_close(o[b, :, h], oracle.output_gate(ro, _pair(z, b, h))[0, :, 0], f"o (b={b}, h={h})")
        assert_close(s[b, h], rs[0, 0], f"final_state (b={b}, h={h})")


def test_full_size_backward_last_window(x):
    """All gradients of the headline shape; the rows of the last W tokens of sampled pairs
    against the oracle's backward over the last W + M tokens from a zero state. The earlier
    tokens reach those rows only through the state at T - W - M, whose effect the decays over
    the M warm-up tokens shrink below the bound the test computes from the data (the reverse
    quantities depend only on later tokens, all inside the window)."""
    W, M = 1024, 1024
    do = ki.gate_logits_like(x["v"], seed=5)
    got = kda.backward(*(x[n] for n in NAMES), do, want_d_initial_state=False)
    kda.check_status()
    for b, h in PAIRS[:2]:
        rows = (T - W - M, T)
        ref = oracle.backward(*(_pair(x[n], b, h, rows) for n in NAMES), _pair(do, b, h, rows))
        a = T - W - M
        bv = (x["beta"][b, :a, h].float() * x["v"][b, :a, h].float().norm(dim=-1)).sum().item()
        log_bound = x["g"][b, a:T - W, h].float().max(dim=-1).values.sum().item() + math.log(max(bv, 1e-30))
        assert log_bound < math.log(1e-12), log_bound
        for name in ("dq", "dk", "dv", "dg"):
            assert_close(got[name][b, T - W:, h], ref[name][0, M:, 0], f"{name} (b={b}, h={h})")
        assert_close(got["dbeta"][b, T - W:, h], ref["dbeta"][0, M:, 0], f"dbeta (b={b}, h={h})")
