"""Backward pass on the GPU (kda_backward): every gradient against the fp64 oracle adjoint
(itself pinned by finite differences), on the same seeded inputs."""

import numpy as np
import pytest
import torch

import gated_delta_rule_56_gb300 as kda
import kda_inputs as ki
import oracle
from kda_testutil import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NAMES = ("q", "k", "v", "g", "beta")
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")


@pytest.fixture(scope="module", autouse=True)
def _built():
    kda.load()


def _check(x, do, dfin=None, cu=None, init=None, rel_frob=None):
    got = kda.backward(*(x[n] for n in NAMES), do, cu_seqlens=cu, initial_state=init, d_final_state=dfin)
    kda.check_status()
    ref = oracle.backward(*(x[n].cpu() for n in NAMES), do.cpu(), None if dfin is None else dfin.cpu(),
                          cu_seqlens=None if cu is None else cu.cpu(), initial_state=None if init is None else init.cpu())
    for name in GRADS:
        if rel_frob is None:
            assert_close(got[name], ref[name], name)
        else:
            assert_close(got[name], ref[name], name, rel_frob=rel_frob)


def _do(x, seed):
    return ki.gate_logits_like(x["v"], seed=seed)  # N(0, 1) entries with the layout and dtype of o


@pytest.mark.parametrize("B,T,H,d,dtype", [(2, 150, 2, 128, torch.bfloat16), (1, 64, 3, 64, torch.float32),
                                           (2, 9, 2, 32, torch.float32), (1, 1, 1, 128, torch.bfloat16)])
def test_backward_matches_oracle(B, T, H, d, dtype):
    x = ki.prefill_inputs(B, T, H, d, d, dtype=dtype, device=DEV, seed=121, state_std=0.02)
    dfin = torch.randn(B, H, d, d, device=DEV, generator=torch.Generator(device=DEV).manual_seed(122))
    _check(x, _do(x, 123), dfin=dfin, init=x["initial_state"])


def test_backward_fp32_inputs_keep_fp32_accuracy():
    """With fp32 inputs the d=128 kernel splits every tensor-core operand (three tf32 products per
    product), so the gradients stay near fp32 rounding: well inside 5e-5 relative, where single tf32
    products (the bf16-input instance) land near 3e-4."""
    x = ki.prefill_inputs(2, 100, 2, 128, 128, dtype=torch.float32, device=DEV, seed=131, state_std=0.02)
    dfin = torch.randn(2, 2, 128, 128, device=DEV, generator=torch.Generator(device=DEV).manual_seed(132))
    _check(x, _do(x, 133), dfin=dfin, init=x["initial_state"], rel_frob=5e-5)


def test_backward_varlen_without_states():
    x = ki.varlen_inputs([70, 1, 130, 64], 2, 128, 128, device=DEV, seed=124)
    _check(x, _do(x, 125), cu=x["cu_seqlens"])


def test_backward_long_memory_across_chunks():
    """Slow decay, so the gradient of early tokens depends on many later ones (several checkpoints)."""
    x = ki.prefill_inputs(1, 300, 2, 64, 64, dtype=torch.float32, device=DEV, seed=126, state_std=0.02)
    x["g"] = x["g"] * 0.01
    _check(x, _do(x, 127), init=x["initial_state"])


def test_backward_varlen_with_empty_sequence_and_states():
    """A zero-length sequence passes its d_final_state straight through as d_initial_state."""
    x = ki.varlen_inputs([33, 0, 17], 2, 128, 128, device=DEV, seed=128)
    dfin = torch.randn(3, 2, 128, 128, device=DEV, generator=torch.Generator(device=DEV).manual_seed(129))
    _check(x, _do(x, 130), dfin=dfin, cu=x["cu_seqlens"], init=x["initial_state"])
    got = kda.backward(*(x[n] for n in NAMES), _do(x, 130), cu_seqlens=x["cu_seqlens"],
                       initial_state=x["initial_state"], d_final_state=dfin)
    kda.check_status()
    assert torch.equal(got["d_initial_state"][1], dfin[1])
