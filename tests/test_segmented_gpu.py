"""Segmented prefill of a few long sequences (split along the sequence, combined through the
segment transitions): parity with the fp64 oracle run over the whole sequences."""

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


def _ws(B, T, H):
    return int(kda.load().kda_prefill_workspace_size(0, B, T, H, 128, 128, None, B))


def _ref(x, init, g=None):
    return oracle.recurrent(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["g"].cpu() if g is None else g,
                            x["beta"].cpu(), initial_state=None if init is None else init.cpu())


def test_workspace_size_for_few_long_sequences():
    # The split depends on the SM count, so the size is asked for on the device. It holds q-tilde
    # (bf16, one row per token-head) plus three 128x128 matrices per (segment, head).
    n = _ws(1, 1 << 20, 32)
    assert n > 0 and n % 256 == 0
    assert n >= (1 << 20) * 32 * 128 * 2
    assert _ws(1, 2048, 2) == 0   # too short to split
    assert _ws(4, 8192, 32) == 0  # enough (sequence, head) pairs to fill the GPU


@pytest.mark.parametrize("B,T,H,with_init", [(1, 8192, 2, False), (1, 8000, 2, True), (2, 6400, 3, True)])
def test_segmented_prefill_matches_oracle(B, T, H, with_init):
    assert _ws(B, T, H) > 0, "this shape should take the segmented path"
    x = ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=51, state_std=0.02 if with_init else None)
    init = x.get("initial_state")
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=init)
    kda.check_status()
    ro, rs = _ref(x, init)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_segmented_prefill_long_memory():
    """Weak decay (g near 0), so each segment's start state matters for its whole length."""
    x = ki.prefill_inputs(1, 8192, 2, 128, 128, device=DEV, seed=52, state_std=0.02)
    x["g"] = (x["g"].float() * 0.002).to(torch.bfloat16)  # log-decays in (-0.01, 0)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = _ref(x, x["initial_state"])
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_segmented_equals_single_pass():
    """Without a workspace the same call takes the single pass; both agree within rounding."""
    x = ki.prefill_inputs(1, 8192, 2, 128, 128, device=DEV, seed=53, state_std=0.02)
    lib = kda.load()
    o1, s1 = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    o2 = torch.empty_like(o1)
    s2 = torch.empty_like(s1)
    st = lib.kda_prefill(0, 1, 8192, 2, 128, 128, *(x[n].data_ptr() for n in NAMES), None, 1,
                         x["initial_state"].data_ptr(), o2.data_ptr(), s2.data_ptr(), None, 0,
                         torch.cuda.current_stream().cuda_stream)
    assert st == 0
    kda.check_status()
    assert (o1.float() - o2.float()).abs().max().item() < 2e-2
    assert ((s1 - s2).norm() / s2.norm()).item() < 5e-3


def test_segmented_gated_prefill():
    x = ki.prefill_inputs(1, 8192, 2, 128, 128, device=DEV, seed=54)
    xg = ki.gate_logits_like(x["g"], seed=55)
    o, s = kda.prefill(x["q"], x["k"], x["v"], xg, x["beta"], gate_bound=5.0)
    kda.check_status()
    ro, rs = _ref(x, None, g=oracle.scaled_sigmoid_gate(xg.cpu(), 5.0))
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_segmented_prefill_mixed_memory():
    """Head 0 decays slowly (its segment transitions stay non-zero, so the transition run covers
    whole segments); head 1 decays fast (its transitions vanish within the first chunks, so the
    run stops early there). Both against the oracle."""
    x = ki.prefill_inputs(1, 8192, 2, 128, 128, device=DEV, seed=56, state_std=0.02)
    g = x["g"].float()
    g[:, :, 0] *= 0.002
    x["g"] = g.to(torch.bfloat16)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = _ref(x, x["initial_state"])
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")
