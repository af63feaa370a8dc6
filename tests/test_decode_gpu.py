"""GPU parity of kda_decode_step against the fp64 oracle (called through the C ABI)."""

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


@pytest.mark.parametrize("dtype,d,N,H", [(torch.bfloat16, 128, 256, 32), (torch.float32, 64, 5, 3),
                                         (torch.bfloat16, 32, 7, 2), (torch.float32, 128, 3, 4)])
def test_decode_step_matches_oracle(dtype, d, N, H):
    """One step on every head (the 256 x 32 x 128 case is the decode workload's shape)."""
    x = ki.decode_inputs(1, N, H, d, d, dtype=dtype, device=DEV, seed=0)
    state = x["state"].clone()
    o = kda.decode_step(*(x[n][0] for n in NAMES), state)
    kda.check_status()
    ro, rs = oracle.decode_step(*(x[n][0].cpu() for n in NAMES), x["state"].cpu())
    assert_close(o, ro, "o")
    assert_close(state, rs, "state")


def test_decode_1000_steps_sampled_heads():
    """1000 consecutive steps of the 256 x 32 x 128 decode workload; sampled heads are
    checked at every step and at the end against the oracle run over the same 1000 tokens."""
    steps, N, H, d = 1000, 256, 32, 128
    x = ki.decode_inputs(steps, N, H, d, d, device=DEV, seed=1)
    state = x["state"].clone()
    sample = [(0, 0), (255, 31), (17, 5), (128, 16), (200, 3), (3, 30)]
    ns = torch.tensor([s[0] for s in sample], device=DEV)
    hs = torch.tensor([s[1] for s in sample], device=DEV)
    outs = torch.empty(steps, len(sample), d, dtype=torch.bfloat16, device=DEV)
    o = torch.empty(N, H, d, dtype=torch.bfloat16, device=DEV)
    for t in range(steps):
        kda.decode_step(*(x[n][t] for n in NAMES), state, o=o)
        outs[t] = o[ns, hs]
    kda.check_status()
    for i, (n, h) in enumerate(sample):
        seq = [x[m][:, n, h].cpu() for m in NAMES]
        seq = [a.reshape(1, steps, 1, *a.shape[1:]) for a in seq]
        ro, rs = oracle.recurrent(*seq, initial_state=x["state"][n, h].reshape(1, 1, d, d).cpu())
        assert_close(outs[:, i], ro[0, :, 0], f"o of (n={n}, h={h})")
        assert_close(state[n, h], rs[0, 0], f"state of (n={n}, h={h})")


def test_decode_empty_batch_is_a_no_op():
    z = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(0, 4, 64, 64, device=DEV)
    o = kda.decode_step(z, z, z, z, torch.zeros(0, 4, dtype=torch.bfloat16, device=DEV), st)
    assert o.shape == (0, 4, 64)
    kda.check_status()
