"""Output gate (o * sigmoid(z)) and the indexed state pool (kda_prefill_ex / kda_decode_step_ex):
parity with the fp64 oracle, and slots the call must not touch left bit for bit."""

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


@pytest.fixture(scope="module", autouse=True)
def _built():
    kda.load()


def _z(like, seed):
    return ki.gate_logits_like(like, seed=seed)  # N(0, 1) entries, shape/dtype/device of `like`


def _ref(x, init=None, g=None, q=None, k=None):
    cu = x.get("cu_seqlens")
    return oracle.recurrent(x["q"].cpu() if q is None else q, x["k"].cpu() if k is None else k, x["v"].cpu(),
                            x["g"].cpu() if g is None else g, x["beta"].cpu(),
                            cu_seqlens=None if cu is None else cu.cpu(),
                            initial_state=None if init is None else init.cpu())


# ------------------------------------------------------------------------- output gate ------

@pytest.mark.parametrize("B,T,H", [(2, 200, 3), (1, 64, 2)])
def test_out_gate_prefill_tensor_core_path(B, T, H):
    x = ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=91, state_std=0.02)
    z = _z(x["v"], seed=92)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], out_gate=z)
    kda.check_status()
    ro, rs = _ref(x, x["initial_state"])
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(s, rs, "final_state")


def test_out_gate_prefill_varlen_ragged_chunks():
    x = ki.varlen_inputs([70, 1, 130, 64], 2, 128, 128, device=DEV, seed=93)
    z = _z(x["v"], seed=94)
    o, s = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"],
                       out_gate=z)
    kda.check_status()
    ro, rs = _ref(x, x["initial_state"])
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(s, rs, "final_state")


def test_out_gate_segmented_long_sequence():
    x = ki.prefill_inputs(1, 8192, 2, 128, 128, device=DEV, seed=95, state_std=0.02)
    assert kda.load().kda_prefill_workspace_size(0, 1, 8192, 2, 128, 128, None, 1) > 0
    z = _z(x["v"], seed=96)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], out_gate=z)
    kda.check_status()
    ro, rs = _ref(x, x["initial_state"])
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(s, rs, "final_state")


def test_out_gate_fp32_recurrent_path_and_decode():
    x = ki.prefill_inputs(2, 50, 2, 64, 64, dtype=torch.float32, device=DEV, seed=97, state_std=0.02)
    z = _z(x["v"], seed=98)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"], out_gate=z)
    kda.check_status()
    ro, rs = _ref(x, x["initial_state"])
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(s, rs, "final_state")
    d = ki.decode_inputs(1, 4, 3, 128, 128, device=DEV, seed=99)
    st = d["state"].clone()
    zd = _z(d["v"][0], seed=100)
    od = kda.decode_step(*(d[n][0] for n in NAMES), st, out_gate=zd)
    kda.check_status()
    rod, rsd = oracle.decode_step(*(d[n][0].cpu() for n in NAMES), d["state"].cpu())
    assert_close(od, oracle.output_gate(rod, zd.cpu()), "o")
    assert_close(st, rsd, "state")


def test_all_options_together():
    """Gate logits, q/k L2 normalisation and the output gate in one call (tensor-core path)."""
    x = ki.prefill_inputs(2, 150, 2, 128, 128, device=DEV, seed=101, state_std=0.02)
    q, k = ki.raw_qk_like(x["q"], seed=102), ki.raw_qk_like(x["k"], seed=103)
    xg, z = ki.gate_logits_like(x["g"], seed=104), _z(x["v"], seed=105)
    o, s = kda.prefill(q, k, x["v"], xg, x["beta"], initial_state=x["initial_state"], gate_bound=5.0,
                       qk_l2norm=True, out_gate=z)
    kda.check_status()
    unit = lambda t: oracle.l2_normalize(t.cpu())  # fp64 normalisation (many tokens: no rounding needed)
    ro, rs = _ref(x, x["initial_state"], g=oracle.scaled_sigmoid_gate(xg.cpu(), 5.0), q=unit(q), k=unit(k))
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(s, rs, "final_state")


# ------------------------------------------------------------------------- state pool -------

def _pool(P, H, d, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn(P, H, d, d, generator=g, device=DEV) * 0.02


@pytest.mark.parametrize("T", [200, 8192])
def test_prefill_reads_and_writes_pool_slots(T):
    B, H, P = (3, 2, 6) if T == 200 else (1, 2, 5)
    x = ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=106)
    pool = _pool(P, H, 128, seed=107)
    before = pool.clone()
    init_idx = torch.tensor([4, -1, 1][:B], dtype=torch.int32, device=DEV)
    fin_idx = torch.tensor([0, 2, 3][:B], dtype=torch.int32, device=DEV)
    o, _ = kda.prefill(*(x[n] for n in NAMES), initial_state=pool, final_state=pool,
                       initial_state_indices=init_idx, final_state_indices=fin_idx)
    kda.check_status()
    init = torch.stack([before[i] if i >= 0 else torch.zeros_like(before[0]) for i in init_idx.tolist()])
    ro, rs = _ref(x, init)
    assert_close(o, ro, "o")
    for n, slot in enumerate(fin_idx.tolist()):
        assert_close(pool[slot], rs[n], f"pool[{slot}]")
    untouched = sorted(set(range(P)) - set(fin_idx.tolist()))
    assert torch.equal(pool[untouched], before[untouched])


def test_decode_pool_in_place_branching_and_inactive():
    N, H, P = 4, 3, 7
    d = ki.decode_inputs(2, N, H, 128, 128, device=DEV, seed=108)
    pool = _pool(P, H, 128, seed=109)
    before = pool.clone()
    idx = torch.tensor([5, 0, -1, 2], dtype=torch.int32, device=DEV)
    o = kda.decode_step(*(d[n][0] for n in NAMES), pool, state_indices=idx)
    kda.check_status()
    init = torch.stack([before[i] if i >= 0 else torch.zeros_like(before[0]) for i in idx.tolist()])
    ro, rs = oracle.decode_step(*(d[n][0].cpu() for n in NAMES), init.cpu())
    assert_close(o, ro, "o")
    for n, slot in enumerate(idx.tolist()):
        if slot >= 0:
            assert_close(pool[slot], rs[n], f"pool[{slot}]")
    assert torch.equal(pool[[1, 3, 4, 6]], before[[1, 3, 4, 6]])  # slots no sequence writes
    # Branch: read slots 5 and 0, write the successors into 6 and 1 (the read slots stay).
    snap = pool.clone()
    src = torch.tensor([5, 0], dtype=torch.int32, device=DEV)
    dst = torch.tensor([6, 1], dtype=torch.int32, device=DEV)
    o2 = kda.decode_step(*(d[n][1][:2] for n in NAMES), pool, state_indices=src, final_state_indices=dst)
    kda.check_status()
    ro2, rs2 = oracle.decode_step(*(d[n][1][:2].cpu() for n in NAMES), snap[[5, 0]].cpu())
    assert_close(o2, ro2, "o")
    assert_close(pool[6], rs2[0], "pool[6]")
    assert_close(pool[1], rs2[1], "pool[1]")
    assert torch.equal(pool[[0, 2, 3, 4, 5]], snap[[0, 2, 3, 4, 5]])


def test_slot_past_the_pool_end_is_reported_and_ignored():
    x = ki.prefill_inputs(2, 64, 2, 128, 128, device=DEV, seed=110)
    pool = _pool(3, 2, 128, seed=111)
    before = pool.clone()
    o, _ = kda.prefill(*(x[n] for n in NAMES), initial_state=pool, final_state=pool,
                       initial_state_indices=torch.tensor([3, 0], dtype=torch.int32, device=DEV),
                       final_state_indices=torch.tensor([1, 7], dtype=torch.int32, device=DEV))
    with pytest.raises(kda.KDAError) as ei:
        kda.check_status()
    assert ei.value.status == 1 and "pool end" in str(ei.value)
    kda.check_status()  # the error word was cleared
    # Sequence 0 started from a zero state (its slot 3 is outside) and wrote slot 1; sequence 1
    # read slot 0 and wrote nothing (slot 7 is outside).
    ro, rs = _ref(x, torch.stack([torch.zeros_like(before[0]), before[0]]))
    assert_close(o, ro, "o")
    assert_close(pool[1], rs[0], "pool[1]")
    assert torch.equal(pool[[0, 2]], before[[0, 2]])
