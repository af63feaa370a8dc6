"""The fp32 chunked prefill on the tensor cores in tf32 (heads of 32 and 64 channels): ragged and
packed sequences, initial states, a state pool, saturated and vanishing gates and slowly decaying
heads, against the fp64 oracle; the options it leaves to the CUDA-core recurrence still give the
oracle's results."""

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


def _ref(x, g=None):
    cu = x.get("cu_seqlens")
    init = x.get("initial_state")
    return oracle.recurrent(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["g"].cpu() if g is None else g,
                            x["beta"].cpu(), cu_seqlens=None if cu is None else cu.cpu(),
                            initial_state=None if init is None else init.cpu())


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("lengths", [[1, 63, 64, 0, 65, 300], [700]])
def test_tf32_packed_sequences_with_states(d, lengths):
    x = ki.varlen_inputs(lengths, 3, d, d, dtype=torch.float32, device=DEV, seed=70 + d)
    o, s = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")
    if 0 in lengths:  # an empty sequence returns its initial state
        i = lengths.index(0)
        torch.testing.assert_close(s[i], x["initial_state"][i], rtol=0, atol=0)


@pytest.mark.parametrize("T", [1, 64, 130])
def test_tf32_batch_ragged_tail(T):
    x = ki.prefill_inputs(2, T, 2, 64, 64, dtype=torch.float32, device=DEV, seed=80 + T, state_std=0.05)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("scale", [0.0, 1.0, "saturated"])
def test_tf32_gate_extremes(scale):
    """No decay (g = 0), the workload's gates, and every gate at the bound (g = -5: the decay
    factors of a chunk span e^320, the range the three reference tiles are built for)."""
    x = ki.prefill_inputs(1, 256, 2, 64, 64, dtype=torch.float32, device=DEV, seed=90)
    x["g"] = torch.full_like(x["g"], -5.0) if scale == "saturated" else x["g"] * scale
    o, s = kda.prefill(*(x[n] for n in NAMES))
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_tf32_slow_decay_long_memory():
    """Log-decays in (-0.01, 0) over 2048 tokens: the state carries its rounding across 32 chunks."""
    x = ki.prefill_inputs(1, 2048, 2, 64, 64, dtype=torch.float32, device=DEV, seed=91, state_std=0.02)
    x["g"] = x["g"] * 0.002
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = _ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_tf32_state_pool():
    """Sequence n reads slot init_idx[n] (negative: zero start) and writes slot fin_idx[n]; the
    other slots are untouched."""
    x = ki.varlen_inputs([100, 70], 2, 64, 64, dtype=torch.float32, device=DEV, seed=92)
    pool = torch.randn(4, 2, 64, 64, device=DEV) * 0.05
    out = pool.clone()
    o, _ = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=pool, final_state=out,
                       initial_state_indices=torch.tensor([2, -1], dtype=torch.int32, device=DEV),
                       final_state_indices=torch.tensor([3, 0], dtype=torch.int32, device=DEV))
    kda.check_status()
    init = torch.stack([pool[2], torch.zeros_like(pool[0])])
    ro, rs = oracle.recurrent(*(x[n].cpu() for n in NAMES), cu_seqlens=x["cu_seqlens"].cpu(), initial_state=init.cpu())
    assert_close(o, ro, "o")
    assert_close(out[3], rs[0], "pool[3]")
    assert_close(out[0], rs[1], "pool[0]")
    for slot in (1, 2):
        torch.testing.assert_close(out[slot], pool[slot], rtol=0, atol=0)


def test_tf32_and_recurrent_paths_agree():
    """The options the tf32 kernel leaves to the CUDA-core recurrence (the output gate) give the
    same outputs as the tf32 kernel times the gate, within the two paths' rounding."""
    x = ki.prefill_inputs(1, 200, 2, 64, 64, dtype=torch.float32, device=DEV, seed=93)
    z = ki.gate_logits_like(x["v"], seed=94)
    o_tc, s_tc = kda.prefill(*(x[n] for n in NAMES))
    o_rec, s_rec = kda.prefill(*(x[n] for n in NAMES), out_gate=z)
    kda.check_status()
    gate = torch.sigmoid(z.double())
    assert ((o_tc.double() * gate - o_rec.double()).norm() / o_rec.double().norm()).item() < 5e-3
    assert ((s_tc - s_rec).norm() / s_rec.norm()).item() < 5e-3
