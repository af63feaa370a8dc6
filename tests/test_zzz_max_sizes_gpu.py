"""Maximum sizes on the GPU: the longest-first launch order at its largest supported count of
packed sequences (4096: the one-CTA bitonic sort's whole shared-memory key array), with empty
sequences among them. Launch order cannot change any result (every (sequence, head) CTA is
independent), so the ordered call must equal the call in index order bit for bit, and both the
fp64 oracle within the parity bar."""

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
    kda.load()


def test_longest_first_order_at_4096_sequences():
    n, H = 4096, 1
    lengths = ki.varlen_lengths(n, 0, 8, seed=61)
    x = ki.varlen_inputs(lengths, H, 128, 128, device=DEV, seed=62)
    lib = kda.load()
    assert lib.kda_prefill_workspace_size(0, 1, int(lengths.sum()), H, 128, 128, x["cu_seqlens"].data_ptr(), n) == n * 4  # ordered
    o1, s1 = kda.prefill(*(x[nm] for nm in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    kda.check_status()
    o2, s2 = torch.empty_like(o1), torch.empty_like(s1)
    st = lib.kda_prefill(0, 1, int(lengths.sum()), H, 128, 128, *(x[nm].data_ptr() for nm in NAMES),
                         x["cu_seqlens"].data_ptr(), n, x["initial_state"].data_ptr(), o2.data_ptr(),
                         s2.data_ptr(), None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    kda.check_status()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)  # launch order changes no bit
    ro, rs = oracle.recurrent(*(x[nm].cpu() for nm in NAMES), cu_seqlens=x["cu_seqlens"].cpu(),
                              initial_state=x["initial_state"].cpu())
    assert_close(o1, ro, "o")
    assert_close(s1, rs, "final_state")
    empty = np.flatnonzero(lengths.numpy() == 0)
    assert empty.size > 0 and torch.equal(s1[empty], x["initial_state"][empty])  # empty: state passes through
