"""q/k L2 normalisation in the kernels (kda_prefill_ex / kda_decode_step_ex with qk_l2norm):
parity with the fp64 oracle fed the oracle's own normalisation of the same raw rows."""

import pytest
import torch

import gated_delta_rule_56_gb300 as kda
import kda_inputs as ki
import oracle
from kda_testutil import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NAMES = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    kda.load()


def _raw(x, seed):
    x = dict(x)
    x["q"] = ki.raw_qk_like(x["q"], seed=seed)
    x["k"] = ki.raw_qk_like(x["k"], seed=seed + 1)
    return x


def _unit(t):
    """The oracle's fp64 normalisation of the raw rows (never rounded: the reference of every
    case is the plain fp64 oracle fed these rows)."""
    return oracle.l2_normalize(t.cpu())


def _ref(x, g=None):
    cu = x.get("cu_seqlens")
    init = x.get("initial_state")
    return oracle.recurrent(_unit(x["q"]), _unit(x["k"]), x["v"].cpu(),
                            x["g"].cpu() if g is None else g, x["beta"].cpu(),
                            cu_seqlens=None if cu is None else cu.cpu(),
                            initial_state=None if init is None else init.cpu())


@pytest.mark.parametrize("B,T,H", [(2, 200, 3), (1, 64, 2), (1, 1, 1), (2, 1, 3)])
def test_l2norm_prefill_tensor_core_path(B, T, H):
    """Ragged, one-chunk and single-token calls. A single token's output is (q.k) beta v plus the
    read-out of the decayed initial state, so it hinges on the cancelling sum q.k: the kernel
    forms it from the raw rows and applies the norms to the fp32 product."""
    x = _raw(ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=71, state_std=0.02), seed=72)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], qk_l2norm=True)
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("seed", [90, 91, 92, 93])
def test_l2norm_single_token_one_head_many_seeds(seed):
    """One token of one head: the relative error of o is that of one scalar, q.k, whatever its
    size. Held to the bar against the unrounded normalisation over several draws."""
    x = _raw(ki.prefill_inputs(1, 1, 1, 128, 128, device=DEV, seed=seed, state_std=0.02), seed=seed + 100)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], qk_l2norm=True)
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_l2norm_prefill_varlen():
    x = _raw(ki.varlen_inputs([70, 1, 130, 64], 2, 128, 128, device=DEV, seed=73), seed=74)
    o, s = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"],
                       qk_l2norm=True)
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_l2norm_with_gate_logits():
    x = _raw(ki.prefill_inputs(2, 150, 2, 128, 128, device=DEV, seed=75), seed=76)
    xg = ki.gate_logits_like(x["g"], seed=77)
    o, s = kda.prefill(x["q"], x["k"], x["v"], xg, x["beta"], gate_bound=5.0, qk_l2norm=True)
    kda.check_status()
    ro, rs = _ref(x, g=oracle.scaled_sigmoid_gate(xg.cpu(), 5.0))
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_l2norm_segmented_long_sequence():
    x = _raw(ki.prefill_inputs(1, 8192, 2, 128, 128, device=DEV, seed=78, state_std=0.02), seed=79)
    assert kda.load().kda_prefill_workspace_size(0, 1, 8192, 2, 128, 128, None, 1) > 0
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], qk_l2norm=True)
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("d", [64, 32])
def test_l2norm_prefill_fp32_recurrent_path(d):
    x = _raw(ki.prefill_inputs(2, 77, 2, d, d, dtype=torch.float32, device=DEV, seed=80, state_std=0.02), seed=81)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], qk_l2norm=True)
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_l2norm_decode_steps():
    N, H, d, steps = 8, 4, 128, 4
    x = ki.decode_inputs(steps, N, H, d, d, device=DEV, seed=82)
    st = x["state"].clone()
    ref_state = x["state"].cpu().double().numpy()
    for t in range(steps):
        q = ki.raw_qk_like(x["q"][t], seed=83 + 2 * t)
        k = ki.raw_qk_like(x["k"][t], seed=84 + 2 * t)
        o = kda.decode_step(q, k, x["v"][t], x["g"][t], x["beta"][t], st, qk_l2norm=True)
        ro, ref_state = oracle.decode_step(_unit(q), _unit(k),
                                           x["v"][t].cpu(), x["g"][t].cpu(), x["beta"][t].cpu(), ref_state)
        kda.check_status()
        assert_close(o, ro, "o")
    assert_close(st, ref_state, "state")


def test_l2norm_is_idempotent_on_unit_rows():
    """Rows that are already unit vectors give what the plain call gives (up to rounding)."""
    x = ki.prefill_inputs(2, 130, 2, 128, 128, device=DEV, seed=85, state_std=0.02)
    o1, s1 = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    o2, s2 = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], qk_l2norm=True)
    kda.check_status()
    assert (o1.float() - o2.float()).abs().max().item() < 2e-2
    assert ((s1 - s2).norm() / s1.norm()).item() < 5e-3
