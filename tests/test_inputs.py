"""The seeded input generator against the input recipe it implements: unit-norm q and k rows,
v ~ N(0, 1), beta = sigmoid(N(0, 1)), log-decays -5 sigmoid(N(0, 1)) per key channel, states
~ N(0, 0.02), sequence lengths uniform on the integers of [lo, hi], and the same tensors for
the same seed."""

import math

import torch

import kda_inputs as ki


def test_prefill_inputs_follow_the_recipe():
    x = ki.prefill_inputs(4, 512, 8, 64, 32, dtype=torch.float32, seed=3, state_std=0.02)
    assert x["q"].shape == (4, 512, 8, 64) and x["v"].shape == (4, 512, 8, 32)
    assert x["beta"].shape == (4, 512, 8) and x["g"].shape == (4, 512, 8, 64)
    assert x["initial_state"].shape == (4, 8, 64, 32) and x["initial_state"].dtype == torch.float32
    for name in ("q", "k"):
        torch.testing.assert_close(x[name].norm(dim=-1), torch.ones(4, 512, 8), rtol=0, atol=1e-5)
    v = x["v"].double()
    assert abs(v.mean().item()) < 0.01 and abs(v.std().item() - 1.0) < 0.01
    b = x["beta"].double()
    assert 0.0 < b.min().item() and b.max().item() < 1.0 and abs(b.mean().item() - 0.5) < 0.01
    g = x["g"].double()
    # sigmoid(N(0,1)) is symmetric about 1/2: E[g] = -2.5; g lies in [-5, 0]
    assert -5.0 <= g.min().item() and g.max().item() <= 0.0 and abs(g.mean().item() + 2.5) < 0.01
    s = x["initial_state"].double()
    assert abs(s.std().item() - 0.02) < 0.0005 and abs(s.mean().item()) < 0.0005


def test_bf16_inputs_are_the_rounded_fp32_draws():
    a = ki.prefill_inputs(1, 64, 2, 128, 128, dtype=torch.float32, seed=11)
    b = ki.prefill_inputs(1, 64, 2, 128, 128, dtype=torch.bfloat16, seed=11)
    for name in ("q", "k", "v", "g", "beta"):
        assert b[name].dtype == torch.bfloat16
        assert torch.equal(b[name], a[name].to(torch.bfloat16)), name
    # the rounded unit rows are unit to bf16 precision only
    err = (b["k"].double().norm(dim=-1) - 1.0).abs().max().item()
    assert 0.0 < err < 2.0 ** -7


def test_same_seed_same_tensors_other_seed_other_tensors():
    a = ki.prefill_inputs(1, 32, 2, 16, 16, seed=5, state_std=0.02)
    b = ki.prefill_inputs(1, 32, 2, 16, 16, seed=5, state_std=0.02)
    c = ki.prefill_inputs(1, 32, 2, 16, 16, seed=6, state_std=0.02)
    for name in ("q", "k", "v", "g", "beta", "initial_state"):
        assert torch.equal(a[name], b[name]), name
        assert not torch.equal(a[name], c[name]), name


def test_varlen_lengths_and_cu_seqlens():
    n = ki.varlen_lengths(4000, 128, 16384, seed=0)
    assert n.dtype == torch.int64 and n.min().item() >= 128 and n.max().item() <= 16384
    assert abs(n.double().mean().item() - (128 + 16384) / 2) < 200  # uniform: mean 8256, sd of mean ~75
    assert torch.equal(n, ki.varlen_lengths(4000, 128, 16384, seed=0))
    tiny = ki.varlen_lengths(2000, 3, 5, seed=1)  # both ends of the range occur
    assert set(tiny.tolist()) == {3, 4, 5}
    cu = ki.cu_seqlens_from_lengths([5, 0, 7])
    assert cu.dtype == torch.int32 and cu.tolist() == [0, 5, 5, 12]
    x = ki.varlen_inputs([5, 0, 7], 2, 16, 8, seed=2)
    assert x["q"].shape == (1, 12, 2, 16) and x["initial_state"].shape == (3, 2, 16, 8)
    assert x["cu_seqlens"].tolist() == [0, 5, 5, 12]


def test_decode_inputs_follow_the_recipe():
    x = ki.decode_inputs(16, 32, 4, 64, 64, dtype=torch.float32, seed=9)
    assert x["q"].shape == (16, 32, 4, 64) and x["beta"].shape == (16, 32, 4)
    assert x["state"].shape == (32, 4, 64, 64)
    torch.testing.assert_close(x["k"].norm(dim=-1), torch.ones(16, 32, 4), rtol=0, atol=1e-5)
    assert abs(x["state"].double().std().item() - ki.STATE_STD) < 0.0005
    g = x["g"].double()
    assert -5.0 <= g.min().item() and g.max().item() <= 0.0


def test_option_draws():
    g = ki.prefill_inputs(2, 256, 4, 64, 64, dtype=torch.float32, seed=1)["g"]
    z = ki.gate_logits_like(g, seed=3)
    assert z.shape == g.shape and z.dtype == g.dtype
    assert abs(z.double().mean().item()) < 0.01 and abs(z.double().std().item() - 1.0) < 0.01
    q = ki.raw_qk_like(g, seed=4)  # rows of 64 N(0,1) entries times exp(U[-1.5, 1.5])
    log_scale = torch.log(q.double().norm(dim=-1) / math.sqrt(64))
    assert log_scale.min().item() > -1.5 - 0.5 and log_scale.max().item() < 1.5 + 0.5
    assert log_scale.max().item() - log_scale.min().item() > 2.5  # the scales spread over the range
