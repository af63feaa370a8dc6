"""Seeded synthetic inputs for KDA prefill and decode.

This module is shared by the CUDA-path tests, the oracle tests and the benchmark. It holds
no KDA arithmetic: only random draws with the distributions of the workloads, namely

* q, k ~ N(0, 1), then L2-normalised over the key dimension for every (token, head),
  in fp32, then rounded to the requested dtype;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1)), one scalar per (token, head);
* log-decay g = -5 * sigmoid(N(0, 1)) for every key channel (the decay bound of 5 keeps
  g in [-5, 0], the range the kernels are accurate on);
* states ~ N(0, 0.02) (standard deviation 0.02) where a workload asks for random states.

Draw order is fixed: q, k, v, beta, g, then states, then sequence lengths. Every function
takes a seed and a device; the same seed on another device gives other (still seeded)
numbers, so a test always hands the very same tensors to both sides of a comparison.
"""

from __future__ import annotations

import torch

DECAY_BOUND = 5.0
STATE_STD = 0.02


def _generator(seed: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def prefill_inputs(B, T, H, dk, dv, dtype=torch.bfloat16, seed=0, device="cpu",
                   n_states=None, state_std=None):
    """Inputs of one prefill call in the [B, T, H, d] layout.

    Returns a dict with q, k [B,T,H,dk], v [B,T,H,dv], g [B,T,H,dk] (all `dtype`),
    beta [B,T,H] (`dtype`) and, when `state_std` is given, an fp32 initial state
    [n_states or B, H, dk, dv].
    """
    gen = _generator(seed, device)
    f32 = dict(generator=gen, device=device, dtype=torch.float32)
    q = torch.randn(B, T, H, dk, **f32)
    k = torch.randn(B, T, H, dk, **f32)
    v = torch.randn(B, T, H, dv, **f32)
    beta = torch.sigmoid(torch.randn(B, T, H, **f32))
    g = -DECAY_BOUND * torch.sigmoid(torch.randn(B, T, H, dk, **f32))
    out = dict(q=_unit(q).to(dtype), k=_unit(k).to(dtype), v=v.to(dtype),
               g=g.to(dtype), beta=beta.to(dtype))
    if state_std is not None:
        n = B if n_states is None else n_states
        out["initial_state"] = torch.randn(n, H, dk, dv, **f32) * float(state_std)
    return out


def gate_logits_like(g: torch.Tensor, seed=0) -> torch.Tensor:
    """Gate logits x ~ N(0, 1) with the shape, dtype and device of a log-decay tensor; the
    log-decay of the workloads is then -5 sigmoid(x)."""
    gen = _generator(seed, g.device)
    return torch.randn(g.shape, generator=gen, device=g.device, dtype=torch.float32).to(g.dtype)


def raw_qk_like(q: torch.Tensor, seed=0) -> torch.Tensor:
    """Un-normalised q or k rows for the in-kernel L2 normalisation: N(0, 1) entries times one
    scale per (token, head) drawn log-uniformly from [e^-1.5, e^1.5], with the shape, dtype and
    device of `q`."""
    gen = _generator(seed, q.device)
    x = torch.randn(q.shape, generator=gen, device=q.device, dtype=torch.float32)
    scale = torch.exp(torch.empty(*q.shape[:-1], 1, device=q.device).uniform_(-1.5, 1.5, generator=gen))
    return (x * scale).to(q.dtype)


def varlen_lengths(n_seqs, lo, hi, seed=0):
    """Sequence lengths drawn uniformly from the integers in [lo, hi]."""
    gen = _generator(seed, "cpu")
    return torch.randint(int(lo), int(hi) + 1, (int(n_seqs),), generator=gen, dtype=torch.int64)


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def varlen_inputs(lengths, H, dk, dv, dtype=torch.bfloat16, seed=0, device="cpu",
                  state_std=STATE_STD):
    """Packed inputs: tensors are [1, sum(lengths), H, d] plus int32 cu_seqlens [N+1]
    and, when `state_std` is not None, one fp32 initial state per sequence."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    total = int(lengths.sum())
    out = prefill_inputs(1, total, H, dk, dv, dtype=dtype, seed=seed, device=device,
                         n_states=lengths.numel(), state_std=state_std)
    out["cu_seqlens"] = cu_seqlens_from_lengths(lengths).to(device)
    return out


def decode_inputs(steps, N, H, dk, dv, dtype=torch.bfloat16, seed=0, device="cpu",
                  state_std=STATE_STD):
    """`steps` consecutive single-token input sets for N sequences, plus an fp32 state.

    q, k, g: [steps, N, H, dk]; v: [steps, N, H, dv]; beta: [steps, N, H];
    state: [N, H, dk, dv] (fp32, N(0, state_std)).
    """
    gen = _generator(seed, device)
    f32 = dict(generator=gen, device=device, dtype=torch.float32)
    q = torch.randn(steps, N, H, dk, **f32)
    k = torch.randn(steps, N, H, dk, **f32)
    v = torch.randn(steps, N, H, dv, **f32)
    beta = torch.sigmoid(torch.randn(steps, N, H, **f32))
    g = -DECAY_BOUND * torch.sigmoid(torch.randn(steps, N, H, dk, **f32))
    state = torch.randn(N, H, dk, dv, **f32) * float(state_std)
    return dict(q=_unit(q).to(dtype), k=_unit(k).to(dtype), v=v.to(dtype), g=g.to(dtype),
                beta=beta.to(dtype), state=state)
