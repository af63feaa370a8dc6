"""Stage-by-stage parity of the tensor-core prefill: the chunkwise intermediates the kernel holds
(Gam, A, T, U and the state at each chunk start), dumped by kda_prefill_debug_dump for the first
(sequence, head), against the oracle's separately written chunkwise form (fp64) on the same inputs.

An end-to-end error says that something is wrong; these comparisons say where. Bars per stage, from
the arithmetic: Gam is an fp32 running sum of bf16 inputs (|Gam| <= 320), so it agrees to about
1e-5 absolute. A, T and U are products of bf16 operands (each factor rounded to 2^-9 relative, T
itself stored in bf16), so about 3e-3 relative (Frobenius) is expected and 1e-2 is the bar, far below
what a wrong index, sign or scale produces (order 1). The state at the chunk starts carries the
prefill's own error, held to the parity bar (5e-3 relative, 2e-2 absolute)."""

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
PER_CHUNK = 40960
GAM, A, T, U, S = 0, 8192, 12288, 16384, 24576


@pytest.fixture(scope="module")
def lib():
    return kda.load()


def _dump(lib, x, T_, H, nch):
    o = torch.empty_like(x["v"])
    fin = torch.empty(1, H, 128, 128, device=DEV)
    d = torch.full((nch * PER_CHUNK,), float("nan"), device=DEV)
    st = lib.kda_prefill_debug_dump(1, T_, H, *(x[n].data_ptr() for n in NAMES), x["initial_state"].data_ptr(),
                                    o.data_ptr(), fin.data_ptr(), d.data_ptr(), nch,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.kda_last_error()
    kda.check_status()
    return o, fin, d.cpu().double().numpy().reshape(nch, PER_CHUNK)


@pytest.mark.parametrize("scale", [1.0, 0.002])
def test_chunkwise_stages_match_the_oracle(lib, scale):
    """Four chunks (the last ragged, 8 rows), an initial state; the workloads' gates and gates 500x
    slower (long memory)."""
    T_, H = 200, 2
    x = ki.prefill_inputs(1, T_, H, 128, 128, device=DEV, seed=91, state_std=0.02)
    x["g"] = (x["g"].float() * scale).to(torch.bfloat16)
    nch = (T_ + 63) // 64
    o, fin, d = _dump(lib, x, T_, H, nch)
    ro, rs, st = oracle.chunked(*(x[n].cpu() for n in NAMES), initial_state=x["initial_state"].cpu(), chunk=64,
                                dump=True)
    # the dump instance computes the same result as the plain call
    assert_close(o, ro, "o")
    assert_close(fin, rs, "final_state")
    og, oa, ou = 0, 0, 0
    for c in range(nch):
        n = min(64, T_ - 64 * c)
        gam = d[c, GAM:GAM + 64 * 128].reshape(64, 128)[:n]
        np.testing.assert_allclose(gam, st["Gam"][og:og + n * 128].reshape(n, 128), rtol=0, atol=1e-4,
                                   err_msg=f"Gam, chunk {c}")
        a = d[c, A:A + 64 * 64].reshape(64, 64)[:n, :n]
        assert_close(a, st["A"][oa:oa + n * n].reshape(n, n), f"A (chunk {c})", max_abs=2e-2, rel_frob=1e-2)
        t = d[c, T:T + 64 * 64].reshape(64, 64)[:n, :n]
        assert_close(t, st["T"][oa:oa + n * n].reshape(n, n), f"T (chunk {c})", max_abs=2e-2, rel_frob=1e-2)
        u = d[c, U:U + 64 * 128].reshape(64, 128)[:n]
        assert_close(u, st["U"][ou:ou + n * 128].reshape(n, 128), f"U (chunk {c})", max_abs=5e-2, rel_frob=1e-2)
        s = d[c, S:S + 128 * 128].reshape(128, 128)
        assert_close(s, st["S_before"][c * 128 * 128:(c + 1) * 128 * 128].reshape(128, 128), f"S (chunk {c})")
        og += n * 128
        oa += n * n
        ou += n * 128
    # the first chunk's state is the initial state exactly (fp32 in, fp32 held)
    np.testing.assert_array_equal(d[0, S:].reshape(128, 128), x["initial_state"][0, 0].double().cpu().numpy())
