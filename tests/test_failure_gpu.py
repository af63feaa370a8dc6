"""Failure detection on the GPU without a GPU fault: a bounded device-side wait that runs out is
reported as KDA_ERR_TIMEOUT and leaves the context usable."""

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


def test_wait_that_runs_out_is_reported_and_context_survives():
    kda.check_status()  # start clean
    kda.selftest_wait_timeout(20_000_000)  # 20 ms on a phase nothing completes
    with pytest.raises(kda.KDAError) as e:
        kda.check_status()
    assert e.value.status == 4 and "KDA_ERR_TIMEOUT" in str(e.value)
    kda.check_status()  # the error word was cleared
    # The same context still runs the tensor-core prefill correctly.
    x = ki.prefill_inputs(1, 130, 2, 128, 128, device=DEV, seed=21, state_std=0.02)
    o, s = kda.prefill(*(x[n] for n in NAMES), initial_state=x["initial_state"])
    kda.check_status()
    ro, rs = oracle.recurrent(*(x[n].cpu() for n in NAMES), initial_state=x["initial_state"].cpu())
    assert_close(o, ro, "o")
    assert_close(s, rs, "final_state")
