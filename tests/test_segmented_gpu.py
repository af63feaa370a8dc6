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


# ---- packed sequences (cu_seqlens): the segments are planned on the device from the lengths ----

def _ws_packed(x, H):
    n = x["cu_seqlens"].numel() - 1
    return int(kda.load().kda_prefill_workspace_size(0, 1, x["q"].shape[1], H, 128, 128,
                                                     x["cu_seqlens"].data_ptr(), n))


def _ref_packed(x, g=None):
    init = x.get("initial_state")
    return oracle.recurrent(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["g"].cpu() if g is None else g,
                            x["beta"].cpu(), cu_seqlens=x["cu_seqlens"].cpu(),
                            initial_state=None if init is None else init.cpu())


def _packed_call_without_workspace(x, H):
    """The same packed call through the C ABI with no workspace: one pass per sequence."""
    lib = kda.load()
    n = x["cu_seqlens"].numel() - 1
    T = x["q"].shape[1]
    o = torch.empty_like(x["v"])
    s = torch.empty(n, H, 128, 128, device=DEV)
    init = x.get("initial_state")
    st = lib.kda_prefill(0, 1, T, H, 128, 128, *(x[m].data_ptr() for m in NAMES), x["cu_seqlens"].data_ptr(), n,
                         None if init is None else init.data_ptr(), o.data_ptr(), s.data_ptr(), None, 0,
                         torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.kda_last_error()
    kda.check_status()
    return o, s


@pytest.mark.parametrize("lengths", [[8192], [100, 9000, 3000, 0, 5000], [4096, 64, 12000]])
def test_packed_split_matches_oracle(lengths):
    """A few packed sequences of mixed lengths (one empty), with initial states: the long ones are
    cut into segments (the first from the sequence's initial state), every output and final state
    against the oracle."""
    H = 2
    x = ki.varlen_inputs(lengths, H, 128, 128, device=DEV, seed=57)
    assert _ws_packed(x, H) > len(lengths) * 4, "these packed sequences should be split"
    o, s = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = _ref_packed(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")
    if 0 in lengths:
        i = lengths.index(0)
        torch.testing.assert_close(s[i], x["initial_state"][i], rtol=0, atol=0)


def test_packed_split_long_memory_and_options():
    """Slowly decaying gates on one head (the transition run then covers whole segments), gate
    logits, q/k L2 normalisation and the output gate together, on split packed sequences."""
    H = 2
    x = ki.varlen_inputs([7000, 300, 9100], H, 128, 128, device=DEV, seed=58)
    assert _ws_packed(x, H) > 256
    xg = ki.gate_logits_like(x["g"], seed=59)
    xg[:, :, 0] = xg[:, :, 0] - 9.0  # -5 sigmoid(x - 9): log-decays near -6e-4 on head 0
    x["q"], x["k"] = ki.raw_qk_like(x["q"], seed=60), ki.raw_qk_like(x["k"], seed=61)
    z = ki.gate_logits_like(x["v"], seed=62)
    o, s = kda.prefill(*(x[n] for n in NAMES[:3]), xg, x["beta"], cu_seqlens=x["cu_seqlens"],
                       initial_state=x["initial_state"], gate_bound=5.0, qk_l2norm=True, out_gate=z)
    kda.check_status()
    xr = dict(x)
    xr["q"], xr["k"] = oracle.l2_normalize(x["q"].cpu()), oracle.l2_normalize(x["k"].cpu())
    ro, rs = oracle.recurrent(xr["q"], xr["k"], x["v"].cpu(), oracle.scaled_sigmoid_gate(xg.cpu(), 5.0), x["beta"].cpu(),
                              cu_seqlens=x["cu_seqlens"].cpu(), initial_state=x["initial_state"].cpu())
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(s, rs, "final_state")


def test_packed_split_state_pool():
    """Packed split with an indexed state pool: sequence n reads slot init_idx[n] (one of them
    negative: zero start) and writes slot fin_idx[n]."""
    H = 2
    x = ki.varlen_inputs([6000, 5000], H, 128, 128, device=DEV, seed=63)
    assert _ws_packed(x, H) > 256
    pool = torch.randn(5, H, 128, 128, device=DEV) * 0.02
    init_idx = torch.tensor([3, -1], dtype=torch.int32, device=DEV)
    fin_idx = torch.tensor([0, 4], dtype=torch.int32, device=DEV)
    out = pool.clone()
    o, _ = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=pool, final_state=out,
                       initial_state_indices=init_idx, final_state_indices=fin_idx)
    kda.check_status()
    init = torch.stack([pool[3], torch.zeros_like(pool[0])])
    ro, rs = oracle.recurrent(*(x[n].cpu() for n in NAMES), cu_seqlens=x["cu_seqlens"].cpu(), initial_state=init.cpu())
    assert_close(o, ro, "o")
    assert_close(out[0], rs[0], "pool[0]")
    assert_close(out[4], rs[1], "pool[4]")
    for slot in (1, 2, 3):  # untouched
        torch.testing.assert_close(out[slot], pool[slot], rtol=0, atol=0)


def test_packed_split_equals_unpacked_split():
    """One packed sequence without an initial state is cut exactly like the same unpacked call (the
    same segments, each run from zero, the same joins), so both give the same bits."""
    H = 2
    x = ki.prefill_inputs(1, 8192, H, 128, 128, device=DEV, seed=64)
    cu = torch.tensor([0, 8192], dtype=torch.int32, device=DEV)
    xp = dict(x, cu_seqlens=cu)
    assert _ws_packed(xp, H) > 256 and _ws(1, 8192, H) > 0
    o1, s1 = kda.prefill(*(x[n] for n in NAMES))
    o2, s2 = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=cu)
    kda.check_status()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_packed_split_agrees_with_single_pass():
    """Without a workspace the packed call runs one pass per sequence; both agree within rounding."""
    H = 2
    x = ki.varlen_inputs([5000, 7000], H, 128, 128, device=DEV, seed=65)
    o1, s1 = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    o2, s2 = _packed_call_without_workspace(x, H)
    assert (o1.float() - o2.float()).abs().max().item() < 2e-2
    assert ((s1 - s2).norm() / s2.norm()).item() < 5e-3
