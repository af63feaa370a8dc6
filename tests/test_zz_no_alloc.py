"""kda_prefill_noalloc: the prefill without a caller workspace, on the library's fixed scratch
array. Its results must equal kda_prefill's with a workspace, call after call."""

import pytest
import torch

import gated_delta_rule_56_gb300 as kda
import kda_inputs as ki

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NAMES = ("q", "k", "v", "g", "beta")
KDA_ERR_UNSUPPORTED = 2


@pytest.fixture(scope="module")
def lib():
    return kda.load()


def _noalloc(lib, x, B, T, H, init):
    o = torch.full_like(x["v"], float("nan"))
    fin = torch.full((B, H, 128, 128), float("nan"), device=DEV)
    st = lib.kda_prefill_noalloc(0, B, T, H, 128, 128, *(x[n].data_ptr() for n in NAMES), None, B,
                                 None if init is None else init.data_ptr(), o.data_ptr(), fin.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    return st, o, fin


@pytest.mark.parametrize("B,T,H", [(1, 8192, 2), (2, 300, 3)])
def test_noalloc_equals_prefill_on_two_calls(lib, B, T, H):
    need = lib.kda_prefill_workspace_size(0, B, T, H, 128, 128, None, B)
    assert need <= lib.kda_prefill_noalloc_capacity()
    if T == 8192:
        assert need > 0, "this shape should be split along the sequence (and use the scratch)"
    for seed in (61, 62):
        x = ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=seed, state_std=0.02)
        init = x["initial_state"]
        o_ref, s_ref = kda.prefill(*(x[n] for n in NAMES), initial_state=init)
        st, o, fin = _noalloc(lib, x, B, T, H, init)
        assert st == 0, lib.kda_last_error()
        kda.check_status()
        assert torch.equal(o, o_ref)
        assert torch.equal(fin, s_ref)


def test_noalloc_rejects_a_call_larger_than_its_scratch(lib):
    B, T, H = 1, 65536, 2
    need = lib.kda_prefill_workspace_size(0, B, T, H, 128, 128, None, B)
    assert need > lib.kda_prefill_noalloc_capacity()
    x = ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=63)
    st, o, _fin = _noalloc(lib, x, B, T, H, None)
    assert st == KDA_ERR_UNSUPPORTED
    assert b"static scratch" in lib.kda_last_error()
    kda.check_status()
    assert torch.isnan(o).all(), "nothing may be queued for a rejected call"


def test_noalloc_packed_sequences_equal_prefill(lib):
    """Packed sequences take their longest-first launch order from the static scratch."""
    x = ki.varlen_inputs([300, 5, 1200, 64], 2, 128, 128, device=DEV, seed=64)
    n = x["cu_seqlens"].numel() - 1
    T = x["q"].shape[1]
    assert 0 < lib.kda_prefill_workspace_size(0, 1, T, 2, 128, 128, x["cu_seqlens"].data_ptr(), n) <= \
        lib.kda_prefill_noalloc_capacity()
    o_ref, s_ref = kda.prefill(*(x[m] for m in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    o = torch.empty_like(o_ref)
    fin = torch.empty_like(s_ref)
    st = lib.kda_prefill_noalloc(0, 1, T, 2, 128, 128, *(x[m].data_ptr() for m in NAMES), x["cu_seqlens"].data_ptr(), n,
                                 x["initial_state"].data_ptr(), o.data_ptr(), fin.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.kda_last_error()
    kda.check_status()
    assert torch.equal(o, o_ref) and torch.equal(fin, s_ref)


def test_noalloc_calls_on_two_streams_are_ordered(lib):
    """Two split calls queued back to back on two different streams share the one scratch array;
    the library orders them on the device (the second waits for the first), so each result
    equals kda_prefill's with a workspace of its own, bit for bit."""
    B, T, H = 1, 8192, 2
    assert lib.kda_prefill_workspace_size(0, B, T, H, 128, 128, None, B) > 0
    xs = [ki.prefill_inputs(B, T, H, 128, 128, device=DEV, seed=s, state_std=0.02) for s in (65, 66)]
    refs = [kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"]) for x in xs]
    outs = [(torch.full_like(x["v"], float("nan")), torch.full((B, H, 128, 128), float("nan"), device=DEV))
            for x in xs]
    torch.cuda.synchronize()  # inputs and the NaN-filled outputs are ready before the side streams run
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for x, (o, fin), s in zip(xs, outs, streams):
        st = lib.kda_prefill_noalloc(0, B, T, H, 128, 128, *(x[n].data_ptr() for n in NAMES), None, B,
                                     x["initial_state"].data_ptr(), o.data_ptr(), fin.data_ptr(), s.cuda_stream)
        assert st == 0, lib.kda_last_error()
    torch.cuda.synchronize()
    kda.check_status()
    for (o, fin), (o_ref, s_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref)
        assert torch.equal(fin, s_ref)
