"""Gate logits in, decays formed in the kernels (kda_prefill_gated, kda_decode_step_gated):
parity with the fp64 oracle fed g = -A sigmoid(x) from the same bf16/fp32 logits."""

import pytest
import torch

import gated_delta_rule_56_gb300 as kda
import kda_inputs as ki
import oracle
from kda_testutil import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
A = 5.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    kda.load()


def _gated(x, seed):
    x = dict(x)
    x["x"] = ki.gate_logits_like(x["g"], seed=seed)
    return x


def _prefill_ref(x, bound=A):
    cu = x.get("cu_seqlens")
    init = x.get("initial_state")
    g = oracle.scaled_sigmoid_gate(x["x"].cpu(), bound)
    return oracle.recurrent(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), g, x["beta"].cpu(),
                            cu_seqlens=None if cu is None else cu.cpu(),
                            initial_state=None if init is None else init.cpu())


@pytest.mark.parametrize("T", [1, 64, 200])
def test_gated_prefill_tensor_core_path(T):
    x = _gated(ki.prefill_inputs(2, T, 2, 128, 128, device=DEV, seed=31, state_std=0.02), seed=32)
    o, s = kda.prefill(x["q"], x["k"], x["v"], x["x"], x["beta"], initial_state=x["initial_state"], gate_bound=A)
    kda.check_status()
    ro, rs = _prefill_ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_gated_prefill_varlen():
    x = _gated(ki.varlen_inputs([70, 1, 130], 2, 128, 128, device=DEV, seed=33), seed=34)
    o, s = kda.prefill(x["q"], x["k"], x["v"], x["x"], x["beta"], cu_seqlens=x["cu_seqlens"],
                       initial_state=x["initial_state"], gate_bound=A)
    kda.check_status()
    ro, rs = _prefill_ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_gated_prefill_fp32_tf32_path():
    """fp32 with gate logits runs the tf32 tensor-core kernel (heads of 64 channels)."""
    x = _gated(ki.prefill_inputs(1, 96, 2, 64, 64, dtype=torch.float32, device=DEV, seed=35, state_std=0.02),
               seed=36)
    o, s = kda.prefill(x["q"], x["k"], x["v"], x["x"], x["beta"], initial_state=x["initial_state"], gate_bound=2.0)
    kda.check_status()
    ro, rs = _prefill_ref(x, bound=2.0)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_gated_decode_step():
    x = ki.decode_inputs(3, 64, 4, 128, 128, device=DEV, seed=37)
    xs = ki.gate_logits_like(x["g"], seed=38)
    st = x["state"].clone()
    ref = x["state"].cpu().double().numpy()
    for t in range(3):
        o = kda.decode_step(x["q"][t], x["k"][t], x["v"][t], xs[t], x["beta"][t], st, gate_bound=A)
        g = oracle.scaled_sigmoid_gate(xs[t].cpu(), A)
        ro, ref = oracle.decode_step(x["q"][t].cpu(), x["k"][t].cpu(), x["v"][t].cpu(), g, x["beta"][t].cpu(), ref)
        kda.check_status()
        assert_close(o, ro, f"o[{t}]")
    assert_close(st, ref, "state")


def test_gated_matches_ungated_on_precomputed_decays():
    """The gated call on logits x equals the plain call on g = -A sigmoid(x) computed in fp32 on
    the host (both on the GPU; the in-kernel gate uses fast fp32 intrinsics)."""
    x = _gated(ki.prefill_inputs(1, 130, 2, 128, 128, dtype=torch.float32, device=DEV, seed=39), seed=40)
    g = -A * torch.sigmoid(x["x"])
    o1, s1 = kda.prefill(x["q"], x["k"], x["v"], x["x"], x["beta"], gate_bound=A)
    o2, s2 = kda.prefill(x["q"], x["k"], x["v"], g, x["beta"])
    kda.check_status()
    torch.testing.assert_close(o1, o2, rtol=1e-4, atol=1e-5)
    torch.testing.assert_close(s1, s2, rtol=1e-4, atol=1e-5)
