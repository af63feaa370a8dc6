"""GPU parity of kda_prefill against the fp64 oracle (called through the C ABI).

Small cases are compared element by element over every output. The full-size workloads
(4 x 8192 x 32 heads; 64 packed sequences of 128..16384 tokens; one 1,048,576-token
sequence) are run whole on the GPU and compared element by element on every (sequence, head)
pair: all outputs and final states of the first two, and for the long sequence the first 32,768
outputs, the outputs around the places where a split call joins segments, and the final state of
every head (the last two against the oracle started 2048 tokens earlier, under a decay bound).
"""

import math

import numpy as np
import pytest
import torch

import gated_delta_rule_56_gb300 as kda
import kda_inputs as ki
import oracle
from kda_testutil import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_56_gb300.build import build
    build()


def run(x, **kw):
    o, s = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x.get("cu_seqlens"),
                       initial_state=x.get("initial_state"), **kw)
    kda.check_status()
    return o, s


def ref(x, **kw):
    cu = x.get("cu_seqlens")
    init = x.get("initial_state")
    return oracle.recurrent(*(x[n].cpu() for n in NAMES), cu_seqlens=None if cu is None else cu.cpu(),
                            initial_state=None if init is None else init.cpu(), **kw)


def pair(x, b, h, rows=None):
    """Inputs of one (batch row, head) as a B=1, H=1 problem (optionally a row range)."""
    sl = slice(None) if rows is None else slice(*rows)
    out = {n: x[n][b:b + 1, sl, h:h + 1].cpu() for n in NAMES}
    return out


def test_fp32_small_head_matches_oracle():
    """fp32 inputs, B=1, T=256, H=2, d=64, zero initial state (the tf32 tensor-core kernel)."""
    x = ki.prefill_inputs(1, 256, 2, 64, 64, dtype=torch.float32, device=DEV, seed=0)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 128, 200])
def test_bf16_d128_matches_oracle(T):
    """bf16, d=128, several chunks and ragged tails, random initial state."""
    x = ki.prefill_inputs(2, T, 3, 128, 128, device=DEV, seed=T, state_std=0.02)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (32, torch.float32), (128, torch.float32)])
def test_other_head_sizes_and_dtypes(d, dtype):
    x = ki.prefill_inputs(2, 100, 2, d, d, dtype=dtype, device=DEV, seed=d, state_std=0.1)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_varlen_small_with_empty_sequence():
    """Packed sequences with lengths 1, 63, 64, 0, 65 and 130: chunks restart at each start,
    an empty sequence returns its initial state."""
    x = ki.varlen_inputs([1, 63, 64, 0, 65, 130], 2, 128, 128, device=DEV, seed=3)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")
    torch.testing.assert_close(s[3], x["initial_state"][3], rtol=0, atol=0)


@pytest.mark.parametrize("lengths", [[100, 20], [64, 5, 64, 3], [70, 1, 57]])
def test_varlen_ragged_chunk_next_to_short_sequence(lengths):
    """A ragged last chunk whose 64-row window reaches into a following short sequence (which
    may end the tensor): every output row must still be that of its own sequence."""
    x = ki.varlen_inputs(lengths, 3, 128, 128, device=DEV, seed=11)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("T", [100, 130])
def test_batch_ragged_tail_next_to_following_row(T):
    """Batched layout with T % 64 != 0: the last chunk of batch row b ends inside the rows of
    batch row b + 1, whose outputs must be left to their own chunks."""
    x = ki.prefill_inputs(3, T, 2, 128, 128, device=DEV, seed=12, state_std=0.02)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


def test_zero_tokens_returns_initial_state():
    x = ki.prefill_inputs(2, 0, 2, 128, 128, device=DEV, seed=4, state_std=0.02)
    o, s = run(x)
    assert o.shape == (2, 0, 2, 128)
    torch.testing.assert_close(s, x["initial_state"], rtol=0, atol=0)


def test_final_state_aliases_initial_state():
    x = ki.prefill_inputs(1, 130, 2, 128, 128, device=DEV, seed=5, state_std=0.02)
    ro, rs = ref(x)
    st = x["initial_state"].clone()
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=st, final_state=st)
    kda.check_status()
    assert s.data_ptr() == st.data_ptr()
    assert_close(o, ro, "o")
    assert_close(st, rs, "final_state")


def test_split_prefill_matches_oracle_on_gpu():
    """Prefill-cache property on the GPU: 300 tokens run as 100 then 200 with the final
    state handed over meets the parity bar against the oracle of the unsplit run (chunk
    boundaries move, so the two GPU runs round differently)."""
    x = ki.prefill_inputs(2, 300, 2, 128, 128, device=DEV, seed=6, state_std=0.02)
    ro, rs = ref(x)
    a = {n: x[n][:, :100].contiguous() for n in NAMES}
    b = {n: x[n][:, 100:].contiguous() for n in NAMES}
    a["initial_state"] = x["initial_state"]
    oa, sa = run(a)
    b["initial_state"] = sa
    ob, sb = run(b)
    assert_close(torch.cat([oa, ob], 1), ro, "o (split run)")
    assert_close(sb, rs, "final_state (split run)")


def test_bad_cu_seqlens_is_reported():
    """A decreasing cu_seqlens is seen by the kernel: that sequence is skipped and
    kda_check_status reports KDA_ERR_INVALID_ARG."""
    x = ki.varlen_inputs([10, 10, 10], 2, 64, 64, device=DEV, seed=7)
    x["cu_seqlens"] = torch.tensor([0, 10, 5, 30], dtype=torch.int32, device=DEV)
    kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    with pytest.raises(kda.KDAError) as e:
        kda.check_status()
    assert e.value.status == 1
    kda.check_status()  # the error word was cleared


def test_full_size_batch_every_pair():
    """B=4, T=8192, H=32, d=128, bf16, zero initial state (the prefill workload): every
    (batch row, head) pair against the oracle, element by element."""
    x = ki.prefill_inputs(4, 8192, 32, 128, 128, device=DEV, seed=0)
    o, s = run(x)
    for b in range(4):
        ro, rs = oracle.recurrent(*(x[n][b:b + 1].cpu() for n in NAMES))
        ob, sb = o[b].cpu(), s[b].cpu()
        for h in range(32):
            assert_close(ob[:, h], ro[0, :, h], f"o (b={b}, h={h})")
            assert_close(sb[h], rs[0, h], f"final_state (b={b}, h={h})")


def test_full_size_varlen_every_pair():
    """64 packed sequences, lengths uniform in [128, 16384] (seed 0), H=32, d=128, bf16,
    initial states ~ N(0, 0.02): every (sequence, head) pair against the oracle."""
    lengths = ki.varlen_lengths(64, 128, 16384, seed=0)
    x = ki.varlen_inputs(lengths, 32, 128, 128, device=DEV, seed=0)
    o, s = run(x)
    cu = x["cu_seqlens"].cpu().long()
    o, s = o.cpu(), s.cpu()
    for n in range(64):
        a, b = int(cu[n]), int(cu[n + 1])
        ro, rs = oracle.recurrent(*(x[m][:, a:b].cpu() for m in NAMES),
                                  initial_state=x["initial_state"][n:n + 1].cpu())
        for h in range(32):
            assert_close(o[0, a:b, h], ro[0, :, h], f"o (seq={n}, h={h})")
            assert_close(s[n, h], rs[0, h], f"final_state (seq={n}, h={h})")


def _decay_bound_log(x, h, lo, hi, start=0):
    """log of a bound on how far the tokens before `lo` can move the state after `hi`: the
    transition of each token has norm <= max_c alpha_c, and from a zero state
    ||S_lo|| <= sum_{t < lo} beta_t ||v_t||. Per head h, from the data."""
    bv = (x["beta"][0, start:lo, h].float() * x["v"][0, start:lo, h].float().norm(dim=-1)).sum().item()
    return x["g"][0, lo:hi, h].float().max(dim=-1).values.sum().item() + math.log(max(bv, 1e-30))


def test_long_context_every_head():
    """B=1, T=1,048,576, H=32, d=128, bf16, every head. Outputs: the first 32,768 tokens
    against the oracle. Final state: the oracle over the last M tokens from a zero state; the
    earlier tokens can move the final state by at most prod_t max_c exp(g_t,c) * ||S_{T-M}||_F,
    which the test computes from the data and requires to be negligible. Outputs where a split
    call joins segments (T/4, T/2, 3T/4): the oracle from a zero state M tokens earlier, under the
    same bound (|o_t| moves by at most that bound times |q_t|). The same tokens passed as one
    packed sequence (cu_seqlens = [0, T], segments planned on the device) are cut into the same
    segments and give the same bits, so every check below holds for both calls."""
    T, H, d, M, P = 1 << 20, 32, 128, 2048, 32768
    x = ki.prefill_inputs(1, T, H, d, d, device=DEV, seed=0)
    o, s = run(x)
    op, sp = run(dict(x, cu_seqlens=torch.tensor([0, T], dtype=torch.int32, device=DEV)))
    assert torch.equal(op, o) and torch.equal(sp, s)
    del op, sp
    ro, _ = oracle.recurrent(*(x[n][:, :P].cpu() for n in NAMES))
    oh = o[0, :P].cpu()
    for h in range(H):
        assert_close(oh[:, h], ro[0, :, h], f"o[:{P}] (h={h})")
    _, rs = oracle.recurrent(*(x[n][:, T - M:].cpu() for n in NAMES))
    sh = s[0].cpu()
    for h in range(H):
        log_bound = _decay_bound_log(x, h, T - M, T)
        assert log_bound < math.log(1e-12), (h, log_bound)
        assert_close(sh[h], rs[0, h], f"final_state (h={h})")
    for R in (T // 4, T // 2, 3 * T // 4):
        a, b = R - 64, R + 512
        rw, _ = oracle.recurrent(*(x[n][:, a - M:b].cpu() for n in NAMES))
        ow = o[0, a:b].cpu()
        for h in range(H):
            log_bound = _decay_bound_log(x, h, a - M, a)
            assert log_bound < math.log(1e-12), (R, h, log_bound)
            assert_close(ow[:, h], rw[0, M:, h], f"o[{a}:{b}] (h={h})")


def test_varlen_longest_first_order_changes_nothing():
    """With the workspace the packed sequences launch longest first; every (sequence, head) is
    computed the same way, so the results equal the natural-order launch bit for bit."""
    x = ki.varlen_inputs([70, 1, 130, 64, 2000, 5, 640], 2, 128, 128, device=DEV, seed=13)
    lib = kda.load()
    n = x["cu_seqlens"].numel() - 1
    assert lib.kda_prefill_workspace_size(0, 1, x["q"].shape[1], 2, 128, 128, x["cu_seqlens"].data_ptr(), n) > 0
    o1, s1 = run(x)
    o2, s2 = torch.empty_like(o1), torch.empty_like(s1)
    st = lib.kda_prefill(0, 1, x["q"].shape[1], 2, 128, 128, *(x[m].data_ptr() for m in NAMES),
                         x["cu_seqlens"].data_ptr(), n, x["initial_state"].data_ptr(), o2.data_ptr(),
                         s2.data_ptr(), None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    kda.check_status()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("d", [128, 64])
def test_more_ctas_than_sms(d):
    """A launch with more (sequence, head) CTAs than the GPU has SMs takes the instance whose
    operand build runs one row per loop iteration: 50 packed sequences (lengths 0..300, ragged
    chunks, one empty) x 4 heads = 200 CTAs, initial states; every output and final state against
    the oracle, and bit for bit against the same sequences run in two launches of fewer CTAs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = 4
    lengths = ki.varlen_lengths(50, 0, 300, seed=23)
    lengths[7] = 0
    assert 50 * H > sms
    x = ki.varlen_inputs(lengths, H, d, d, device=DEV, seed=24)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")
    # The first 25 sequences alone (100 CTAs): the two-row instance; same bits.
    cut = int(lengths[:25].sum())
    x1 = {n: x[n][:, :cut] for n in NAMES}
    x1["cu_seqlens"] = x["cu_seqlens"][:26].clone()
    x1["initial_state"] = x["initial_state"][:25]
    assert 25 * H <= sms
    o1, s1 = run(x1)
    assert torch.equal(o1, o[:, :cut]) and torch.equal(s1, s[:25])


@pytest.mark.parametrize("d", [64, 32])
@pytest.mark.parametrize("lengths", [[200], [70, 1, 130, 0, 64, 2000]])
def test_small_heads_bf16_tensor_core_path(d, lengths):
    """bf16 heads of 64 or 32 channels run the tensor-core kernel with the missing channels zero:
    ragged chunks, packed sequences (one empty), initial states, every output and final state."""
    x = ki.varlen_inputs(lengths, 3, d, d, device=DEV, seed=14 + d)
    o, s = run(x)
    ro, rs = ref(x)
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")


@pytest.mark.parametrize("d", [64, 32])
def test_small_heads_bf16_with_options(d):
    """Gate logits, q/k L2 normalisation, the output gate and a state pool on 64/32-channel heads."""
    H = 2
    x = ki.varlen_inputs([150, 70], H, d, d, device=DEV, seed=16 + d)
    xg = ki.gate_logits_like(x["g"], seed=18)
    q, k = ki.raw_qk_like(x["q"], seed=19), ki.raw_qk_like(x["k"], seed=20)
    z = ki.gate_logits_like(x["v"], seed=21)
    pool = torch.randn(4, H, d, d, device=DEV) * 0.02
    out = pool.clone()
    idx_in = torch.tensor([2, -1], dtype=torch.int32, device=DEV)
    idx_out = torch.tensor([0, 3], dtype=torch.int32, device=DEV)
    o, _ = kda.prefill(q, k, x["v"], xg, x["beta"], cu_seqlens=x["cu_seqlens"], initial_state=pool, final_state=out,
                       gate_bound=5.0, qk_l2norm=True, out_gate=z, initial_state_indices=idx_in,
                       final_state_indices=idx_out)
    kda.check_status()
    init = torch.stack([pool[2], torch.zeros_like(pool[0])])
    ro, rs = oracle.recurrent(oracle.l2_normalize(q.cpu()), oracle.l2_normalize(k.cpu()), x["v"].cpu(),
                              oracle.scaled_sigmoid_gate(xg.cpu(), 5.0), x["beta"].cpu(),
                              cu_seqlens=x["cu_seqlens"].cpu(), initial_state=init.cpu())
    assert_close(o, oracle.output_gate(ro, z.cpu()), "o")
    assert_close(out[0], rs[0], "pool[0]")
    assert_close(out[3], rs[1], "pool[3]")
    torch.testing.assert_close(out[1], pool[1], rtol=0, atol=0)
    torch.testing.assert_close(out[2], pool[2], rtol=0, atol=0)
