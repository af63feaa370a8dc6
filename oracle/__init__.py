"""fp64 CPU oracle for Kimi Delta Attention (KDA) -- test infrastructure.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
package. It does not import the CUDA package, and the CUDA package does not import it.
The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, OpenMP over (sequence, head));
this module only builds it with gcc, marshals arrays and calls it.

Public functions take CPU tensors or arrays in the KDA layouts and return fp64 numpy arrays:

* ``recurrent(q, k, v, g, beta, cu_seqlens=None, initial_state=None)`` -> (o, final_state)
* ``literal(...)``: same, with the d_k x d_k transition formed explicitly (small cases)
* ``chunked(..., chunk=64, dump=False)`` -> (o, final_state[, intermediates])
* ``decode_step(q, k, v, g, beta, state)`` -> (o, new_state): one token of the recurrence.
* ``scaled_sigmoid_gate(x, bound)`` -> g = -bound * sigmoid(x) (log-decays from gate logits).
* ``l2_normalize(x, eps=1e-6)`` -> rows along the last axis divided by sqrt(sum x^2 + eps).
* ``output_gate(o, z)`` -> o * sigmoid(z) (the output gate).
* ``backward(q, k, v, g, beta, d_o, d_final_state=None, ...)`` -> gradients (dict) of
  sum(d_o * o) + sum(d_final_state * final_state).

Layouts: q, k, g [B, T, H, d_k]; v [B, T, H, d_v]; beta [B, T, H]; with ``cu_seqlens``
(int [N+1]) B must be 1 and the rows of sequence n are cu[n]..cu[n+1]-1. States are
[N, H, d_k, d_v]. Values are widened to fp64 exactly (bf16 and fp32 both embed in fp64).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (-O2, IEEE semantics, OpenMP). Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    lib.kda_oracle_scaled_sigmoid_gate.argtypes = [ctypes.c_int64, _dp, ctypes.c_double, _dp]
    lib.kda_oracle_scaled_sigmoid_gate.restype = ctypes.c_int
    lib.kda_oracle_backward.argtypes = [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
    lib.kda_oracle_backward.restype = ctypes.c_int
    lib.kda_oracle_output_gate.argtypes = [ctypes.c_int64, _dp, _dp, _dp]
    lib.kda_oracle_output_gate.restype = ctypes.c_int
    lib.kda_oracle_l2_normalize.argtypes = [ctypes.c_int64, ctypes.c_int64, _dp, ctypes.c_double, _dp]
    lib.kda_oracle_l2_normalize.restype = ctypes.c_int
    lib.kda_oracle_recurrent.argtypes = [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
    lib.kda_oracle_recurrent.restype = ctypes.c_int
    lib.kda_oracle_literal.argtypes = [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
    lib.kda_oracle_literal.restype = ctypes.c_int
    lib.kda_oracle_chunked.argtypes = [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                       _dp, _dp, _dp, _dp, _dp]
    lib.kda_oracle_chunked.restype = ctypes.c_int
    lib.kda_oracle_max_threads.argtypes = []
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library; a path loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


class use_library:
    """Context manager: route this module's calls through another build of the oracle
    (used by the test that plants mistakes in a copy of the C source)."""

    def __init__(self, path: str):
        self.lib = _declare(ctypes.CDLL(path))

    def __enter__(self):
        global _lib
        load_library()
        self.saved, _lib = _lib, self.lib
        return self.lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def max_threads() -> int:
    return int(load_library().kda_oracle_max_threads())


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen on the torch side (bf16 has no numpy dtype)
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _flatten(q, k, v, g, beta, cu_seqlens):
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("inconsistent shapes")
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("bad cu_seqlens")
    flat = lambda a, d: a.reshape(B * T, H, d) if d else a.reshape(B * T, H)
    return (flat(q, dk), flat(k, dk), flat(v, dv), flat(g, dk), flat(beta, None), cu, B, T, H, dk, dv)


def _run(kind, q, k, v, g, beta, cu_seqlens=None, initial_state=None, n_threads=0, chunk=64,
         dump=False):
    q, k, v, g, beta, cu, B, T, H, dk, dv = _flatten(q, k, v, g, beta, cu_seqlens)
    N = cu.size - 1
    init = _f64(initial_state)
    if init is not None and init.shape != (N, H, dk, dv):
        raise ValueError(f"initial_state must be {(N, H, dk, dv)}, got {init.shape}")
    o = np.zeros((B * T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64)
    lib = load_library()
    common = (ctypes.c_int(N), cu.ctypes.data_as(_i64p), H, dk, dv)
    tensors = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init), _ptr(o), _ptr(fin))
    extra = None
    if kind == "recurrent":
        rc = lib.kda_oracle_recurrent(*common, *tensors, int(n_threads))
    elif kind == "literal":
        rc = lib.kda_oracle_literal(*common, *tensors)
    else:
        if dump:
            L0 = int(cu[1] - cu[0]) if N else 0
            nch = -(-L0 // chunk)
            extra = dict(Gam=np.zeros(L0 * dk), A=np.zeros(L0 * chunk), T=np.zeros(L0 * chunk),
                         U=np.zeros(L0 * dv), S_before=np.zeros(nch * dk * dv))
            dptr = [_ptr(extra[n]) for n in ("Gam", "A", "T", "U", "S_before")]
        else:
            dptr = [None] * 5
        rc = lib.kda_oracle_chunked(*common, int(chunk), *tensors, int(n_threads), *dptr)
    if rc != 0:
        raise RuntimeError(f"oracle {kind} failed with code {rc}")
    o = o.reshape(B, T, H, dv)
    return (o, fin, extra) if dump else (o, fin)


def recurrent(q, k, v, g, beta, cu_seqlens=None, initial_state=None, n_threads=0):
    """The token recurrence; returns (o [B,T,H,dv], final_state [N,H,dk,dv]) in fp64."""
    return _run("recurrent", q, k, v, g, beta, cu_seqlens, initial_state, n_threads)


def literal(q, k, v, g, beta, cu_seqlens=None, initial_state=None):
    """The recurrence with an explicit d_k x d_k transition per token (small cases)."""
    return _run("literal", q, k, v, g, beta, cu_seqlens, initial_state)


def chunked(q, k, v, g, beta, cu_seqlens=None, initial_state=None, chunk=64, n_threads=0,
            dump=False):
    """The chunkwise form; with dump=True also returns per-chunk intermediates of the
    first (sequence, head) pair (flat fp64 arrays, chunk after chunk)."""
    return _run("chunked", q, k, v, g, beta, cu_seqlens, initial_state, n_threads, chunk, dump)


def backward(q, k, v, g, beta, d_o, d_final_state=None, cu_seqlens=None, initial_state=None):
    """Gradients of L = sum(d_o * o) + sum(d_final_state * final_state) through the recurrence.
    Returns a dict of fp64 arrays: dq, dk, dg [B,T,H,dk], dv [B,T,H,dv], dbeta [B,T,H] and
    d_initial_state [N,H,dk,dv] (the gradient with respect to the initial state, zeros or not)."""
    q, k, v, g, beta, cu, B, T, H, dk, dv = _flatten(q, k, v, g, beta, cu_seqlens)
    N = cu.size - 1
    init = _f64(initial_state)
    if init is not None and init.shape != (N, H, dk, dv):
        raise ValueError(f"initial_state must be {(N, H, dk, dv)}, got {init.shape}")
    do = _f64(d_o).reshape(B * T, H, dv)
    dfin = _f64(d_final_state)
    if dfin is not None and dfin.shape != (N, H, dk, dv):
        raise ValueError(f"d_final_state must be {(N, H, dk, dv)}, got {dfin.shape}")
    out = dict(dq=np.zeros((B * T, H, dk)), dk=np.zeros((B * T, H, dk)), dv=np.zeros((B * T, H, dv)),
               dg=np.zeros((B * T, H, dk)), dbeta=np.zeros((B * T, H)), d_initial_state=np.zeros((N, H, dk, dv)))
    rc = load_library().kda_oracle_backward(
        ctypes.c_int(N), cu.ctypes.data_as(_i64p), H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(init), _ptr(do), _ptr(dfin), *(_ptr(out[n]) for n in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")))
    if rc != 0:
        raise RuntimeError(f"oracle backward failed with code {rc}")
    for n, d in (("dq", dk), ("dk", dk), ("dg", dk), ("dv", dv)):
        out[n] = out[n].reshape(B, T, H, d)
    out["dbeta"] = out["dbeta"].reshape(B, T, H)
    return out


def scaled_sigmoid_gate(x, bound):
    """Log-decays from gate logits: g = -bound * sigmoid(x) elementwise, fp64, same shape as x."""
    x = _f64(x)
    g = np.empty_like(x)
    rc = load_library().kda_oracle_scaled_sigmoid_gate(x.size, x.ctypes.data_as(_dp), float(bound), g.ctypes.data_as(_dp))
    if rc != 0:
        raise ValueError(f"kda_oracle_scaled_sigmoid_gate returned {rc}")
    return g


def output_gate(o, z):
    """o * sigmoid(z) elementwise, fp64, shape of o (z must have the same shape)."""
    o, z = _f64(o), _f64(z)
    if o.shape != z.shape:
        raise ValueError(f"output_gate: shapes {o.shape} and {z.shape} differ")
    y = np.empty_like(o)
    rc = load_library().kda_oracle_output_gate(o.size, o.ctypes.data_as(_dp), z.ctypes.data_as(_dp), y.ctypes.data_as(_dp))
    if rc != 0:
        raise ValueError(f"kda_oracle_output_gate returned {rc}")
    return y


def l2_normalize(x, eps=1e-6):
    """Each row along the last axis divided by sqrt(sum of squares + eps), fp64, same shape."""
    x = _f64(x)
    y = np.empty_like(x)
    d = x.shape[-1] if x.ndim else 0
    rows = x.size // d if d else 0
    rc = load_library().kda_oracle_l2_normalize(rows, d, x.ctypes.data_as(_dp), float(eps), y.ctypes.data_as(_dp))
    if rc != 0:
        raise ValueError(f"kda_oracle_l2_normalize returned {rc}")
    return y


def decode_step(q, k, v, g, beta, state, n_threads=0):
    """One decode token. q, k, g [N,H,dk]; v [N,H,dv]; beta [N,H]; state [N,H,dk,dv].
    Returns (o [N,H,dv], new_state) in fp64."""
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    N, H, dk = q.shape
    dv = v.shape[-1]
    add_t = lambda a: a.reshape(N, 1, *a.shape[1:])
    cu = np.arange(N + 1, dtype=np.int64)
    o, fin = recurrent(add_t(q).reshape(1, N, H, dk), add_t(k).reshape(1, N, H, dk),
                       add_t(v).reshape(1, N, H, dv), add_t(g).reshape(1, N, H, dk),
                       beta.reshape(1, N, H), cu_seqlens=cu, initial_state=state,
                       n_threads=n_threads)
    return o.reshape(N, H, dv), fin
