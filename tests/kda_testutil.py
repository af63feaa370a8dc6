"""Helpers shared by the GPU parity tests: tolerances and comparison against the oracle."""

import json
import os

import numpy as np
import torch

# Parity bar for bf16/fp32 inputs with an fp32 state: per tensor, max-abs error <= 2e-2 and
# relative Frobenius error <= 5e-3 against the fp64 oracle.
MAX_ABS = 2e-2
REL_FROB = 5e-3


def to64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got, ref):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    d = got - ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    denom = float(np.linalg.norm(ref.ravel()))
    rel = float(np.linalg.norm(d.ravel()) / denom) if denom > 0 else float(np.linalg.norm(d.ravel()))
    return max_abs, rel


def _log(name, ma, rf):
    """Append the measured errors to $KDA_PARITY_LOG (JSON lines) when it is set."""
    path = os.environ.get("KDA_PARITY_LOG")
    if path:
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        with open(path, "a") as f:
            f.write(json.dumps({"test": test, "tensor": name, "max_abs": ma, "rel_frob": rf}) + "\n")


def assert_close(got, ref, name, max_abs=MAX_ABS, rel_frob=REL_FROB):
    ma, rf = errors(got, ref)
    _log(name, ma, rf)
    assert ma <= max_abs and rf <= rel_frob, f"{name}: max-abs {ma:.3e} (<= {max_abs}), rel-Frob {rf:.3e} (<= {rel_frob})"
    return ma, rf


def cpu(x):
    return {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in x.items()}
