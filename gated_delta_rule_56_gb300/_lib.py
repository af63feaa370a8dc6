"""ctypes binding of libkda.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels. This module checks the
torch tensors it is handed (device, dtype, shape, contiguity), allocates the outputs the
caller did not pass, and forwards raw device pointers and the current CUDA stream to the
C ABI declared in include/kda.h. There is no fallback: without the built library the
functions raise.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from .build import LIB_PATH, INCLUDE

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_BF16, KDA_F32 = 0, 1
_DTYPES = {torch.bfloat16: KDA_BF16, torch.float32: KDA_F32}


class KDAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int


def library_path() -> str:
    return LIB_PATH


def declared_symbols() -> list[str]:
    """Names of the functions include/kda.h declares."""
    text = open(os.path.join(INCLUDE, "kda.h")).read()
    return re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)


def load():
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first with "
                               "gated_delta_rule_56_gb300.build.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        lib.kda_prefill.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp,
                                    _vp, _vp, ctypes.c_size_t, _vp]
        lib.kda_prefill.restype = _i
        lib.kda_prefill_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _i]
        lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
        lib.kda_prefill_workspace_size_for.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _i, _i]
        lib.kda_prefill_workspace_size_for.restype = ctypes.c_size_t
        lib.kda_prefill_split_plan.argtypes = [_i, _i, _i, _i, _vp, _vp, _vp]
        lib.kda_prefill_split_plan.restype = _i
        lib.kda_decode_step.argtypes = [_i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        lib.kda_decode_step.restype = _i
        lib.kda_check_status.argtypes = [_vp]
        lib.kda_check_status.restype = _i
        lib.kda_status_string.argtypes = [_i]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        lib.kda_version.restype = _i
        lib.kda_prefill_gated.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp,
                                          _vp, ctypes.c_float, _vp, ctypes.c_size_t, _vp]
        lib.kda_prefill_gated.restype = _i
        lib.kda_decode_step_gated.argtypes = [_i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                              ctypes.c_float, _vp]
        lib.kda_decode_step_gated.restype = _i
        lib.kda_prefill_ex.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp,
                                       _vp, ctypes.POINTER(KDAOptions), _vp, ctypes.c_size_t, _vp]
        lib.kda_prefill_ex.restype = _i
        lib.kda_decode_step_ex.argtypes = [_i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                           ctypes.POINTER(KDAOptions), _vp]
        lib.kda_decode_step_ex.restype = _i
        lib.kda_backward.argtypes = [_i, _i, _i, _i, _i, _i] + [_vp] * 6 + [_i] + [_vp] * 10 + [ctypes.c_size_t, _vp]
        lib.kda_backward.restype = _i
        lib.kda_backward_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
        lib.kda_backward_workspace_size.restype = ctypes.c_size_t
        lib.kda_prefill_noalloc.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp,
                                            _vp, _vp, _vp]
        lib.kda_prefill_noalloc.restype = _i
        lib.kda_prefill_noalloc_capacity.argtypes = []
        lib.kda_prefill_noalloc_capacity.restype = ctypes.c_size_t
        lib.kda_prefill_debug_dump.argtypes = [_i, _i, _i] + [_vp] * 8 + [_vp, _i, _vp]
        lib.kda_prefill_debug_dump.restype = _i
        lib.kda_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp]
        lib.kda_selftest_wait_timeout.restype = _i
        _lib = lib
        return lib


class KDAOptions(ctypes.Structure):
    """kda_options of include/kda.h (struct_size first; zero fields are the defaults)."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("gate_bound", ctypes.c_float), ("qk_l2norm", ctypes.c_int),
                ("initial_state_indices", ctypes.c_void_p), ("final_state_indices", ctypes.c_void_p),
                ("state_pool_size", ctypes.c_int), ("out_gate", ctypes.c_void_p)]


def _options(gate_bound, qk_l2norm, init_idx=None, fin_idx=None, pool=0, out_gate=None):
    return KDAOptions(ctypes.sizeof(KDAOptions), 0.0 if gate_bound is None else float(gate_bound),
                      1 if qk_l2norm else 0, None if init_idx is None else init_idx.data_ptr(),
                      None if fin_idx is None else fin_idx.data_ptr(), int(pool),
                      None if out_gate is None else out_gate.data_ptr())


def _check_indices(name, idx, n, dev):
    if idx is not None:
        _check(name, idx, torch.int32, (n,), dev)


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def last_error() -> str:
    return load().kda_last_error().decode()


def version() -> int:
    return int(load().kda_version())


def _raise_if(status: int):
    if status != KDA_OK:
        raise KDAError(status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(name, t, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill(q, k, v, g, beta, cu_seqlens=None, initial_state=None, output_final_state=True,
            o=None, final_state=None, gate_bound=None, qk_l2norm=False, initial_state_indices=None,
            final_state_indices=None, out_gate=None):
    """Chunked KDA prefill on the GPU.

    q, k, g [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H]; all bf16 or all fp32, on one CUDA
    device. With ``cu_seqlens`` (int32 [N+1] on the device) B must be 1 and the rows are
    packed sequences. ``initial_state``: fp32 [N, H, dk, dv] or None (zeros). With
    ``gate_bound`` A, ``g`` holds gate logits x and the kernels use g = -A * sigmoid(x)
    (kda_prefill_gated). With ``qk_l2norm`` the kernels divide every row of q and k by
    sqrt(sum x^2 + 1e-6) (kda_prefill_ex). With ``initial_state_indices`` / ``final_state_indices``
    (int32 [N] on the device) the matching state tensor is a pool [P, H, dk, dv] and sequence n
    reads / writes slot idx[n] (negative: zero start / no write); ``final_state`` must then be
    given. With ``out_gate`` z (the layout and dtype of o) the kernels store o * sigmoid(z).
    Returns (o [B, T, H, dv], final_state [N, H, dk, dv] fp32 (or the pool) or None).
    """
    lib = load()
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for name, t, shp in (("q", q, (B, T, H, dk)), ("k", k, (B, T, H, dk)), ("g", g, (B, T, H, dk)),
                         ("v", v, (B, T, H, dv)), ("beta", beta, (B, T, H))):
        _check(name, t, q.dtype, shp, dev)
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a 1-D int32 tensor [N+1]")
        _check("cu_seqlens", cu_seqlens, torch.int32, (cu_seqlens.numel(),), dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    pools = [t.shape[0] for t, i in ((initial_state, initial_state_indices), (final_state, final_state_indices))
             if t is not None and i is not None and t.dim() == 4]
    if len(set(pools)) > 1:
        raise ValueError("initial and final state pools must have the same number of slots")
    pool = pools[0] if pools else 0
    _check_indices("initial_state_indices", initial_state_indices, N, dev)
    _check_indices("final_state_indices", final_state_indices, N, dev)
    if initial_state is not None:
        n0 = pool if initial_state_indices is not None else N
        _check("initial_state", initial_state, torch.float32, (n0, H, dk, dv), dev)
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=q.dtype, device=dev)
    else:
        _check("o", o, q.dtype, (B, T, H, dv), dev)
    if final_state_indices is not None and final_state is None:
        raise ValueError("final_state_indices needs final_state (the pool)")
    if out_gate is not None:
        _check("out_gate", out_gate, q.dtype, (B, T, H, dv), dev)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    elif final_state is not None:
        n1 = pool if final_state_indices is not None else N
        _check("final_state", final_state, torch.float32, (n1, H, dk, dv), dev)
    dt = _DTYPES[q.dtype]
    ws_bytes = int(lib.kda_prefill_workspace_size(dt, B, T, H, dk, dv, _ptr(cu_seqlens), N))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    with torch.cuda.device(dev):
        if (qk_l2norm or initial_state_indices is not None or final_state_indices is not None
                or out_gate is not None):
            opt = _options(gate_bound, qk_l2norm, initial_state_indices, final_state_indices, pool, out_gate)
            st = lib.kda_prefill_ex(dt, B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(cu_seqlens), N, _ptr(initial_state), _ptr(o), _ptr(final_state),
                                    ctypes.byref(opt), _ptr(ws), ws_bytes, _stream(dev))
        elif gate_bound is None:
            st = lib.kda_prefill(dt, B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 _ptr(cu_seqlens), N, _ptr(initial_state), _ptr(o), _ptr(final_state),
                                 _ptr(ws), ws_bytes, _stream(dev))
        else:
            st = lib.kda_prefill_gated(dt, B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                       _ptr(cu_seqlens), N, _ptr(initial_state), _ptr(o), _ptr(final_state),
                                       float(gate_bound), _ptr(ws), ws_bytes, _stream(dev))
    _raise_if(st)
    return o, final_state


def decode_step(q, k, v, g, beta, state, o=None, gate_bound=None, qk_l2norm=False, state_indices=None,
                final_state_indices=None, out_gate=None):
    """One KDA decode token for N sequences; ``state`` (fp32 [N, H, dk, dv]) is updated in
    place. q, k, g [N, H, dk]; v [N, H, dv]; beta [N, H]. With ``gate_bound`` A, ``g`` holds gate
    logits x and g = -A * sigmoid(x) is used (kda_decode_step_gated). With ``qk_l2norm`` the
    rows of q and k are L2-normalised in the kernel (kda_decode_step_ex). With ``state_indices``
    (int32 [N] on the device) ``state`` is a pool [P, H, dk, dv]: sequence n reads slot
    state_indices[n] (negative: zero state) and writes slot final_state_indices[n] (default: the
    same slot; negative: not written). With ``out_gate`` z [N, H, dv] the kernel stores
    o * sigmoid(z). Returns o [N, H, dv]."""
    lib = load()
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    N, H, dk = q.shape
    dv = v.shape[-1]
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("g", g, (N, H, dk)),
                         ("v", v, (N, H, dv)), ("beta", beta, (N, H))):
        _check(name, t, q.dtype, shp, dev)
    if final_state_indices is not None and state_indices is None:
        raise ValueError("final_state_indices needs state_indices")
    _check_indices("state_indices", state_indices, N, dev)
    _check_indices("final_state_indices", final_state_indices, N, dev)
    pool = state.shape[0] if state_indices is not None and state.dim() == 4 else 0
    _check("state", state, torch.float32, (pool if state_indices is not None else N, H, dk, dv), dev)
    if out_gate is not None:
        _check("out_gate", out_gate, q.dtype, (N, H, dv), dev)
    if o is None:
        o = torch.empty(N, H, dv, dtype=q.dtype, device=dev)
    else:
        _check("o", o, q.dtype, (N, H, dv), dev)
    with torch.cuda.device(dev):
        if qk_l2norm or state_indices is not None or out_gate is not None:
            opt = _options(gate_bound, qk_l2norm, state_indices, final_state_indices, pool, out_gate)
            st = lib.kda_decode_step_ex(_DTYPES[q.dtype], N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(state), _ptr(o), ctypes.byref(opt), _stream(dev))
        elif gate_bound is None:
            st = lib.kda_decode_step(_DTYPES[q.dtype], N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                     _ptr(beta), _ptr(state), _ptr(o), _stream(dev))
        else:
            st = lib.kda_decode_step_gated(_DTYPES[q.dtype], N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                           _ptr(beta), _ptr(state), _ptr(o), float(gate_bound), _stream(dev))
    _raise_if(st)
    return o


def backward(q, k, v, g, beta, d_o, cu_seqlens=None, initial_state=None, d_final_state=None,
             want_d_initial_state=True):
    """Gradients of sum(d_o * o) + sum(d_final_state * final_state) through ``prefill`` (plain
    log-decays g). Inputs as ``prefill``; d_o has the layout and dtype of o; d_final_state fp32
    [N, H, dk, dv] or None. Returns a dict of fp32 tensors: dq, dk, dg [B, T, H, dk], dv
    [B, T, H, dv], dbeta [B, T, H] and d_initial_state [N, H, dk, dv] (or None)."""
    lib = load()
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for name, t, shp in (("q", q, (B, T, H, dk)), ("k", k, (B, T, H, dk)), ("g", g, (B, T, H, dk)),
                         ("v", v, (B, T, H, dv)), ("beta", beta, (B, T, H)), ("d_o", d_o, (B, T, H, dv))):
        _check(name, t, q.dtype, shp, dev)
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a 1-D int32 tensor [N+1]")
        _check("cu_seqlens", cu_seqlens, torch.int32, (cu_seqlens.numel(),), dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _check(name, t, torch.float32, (N, H, dk, dv), dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(dq=torch.empty(B, T, H, dk, **f32), dk=torch.empty(B, T, H, dk, **f32),
               dv=torch.empty(B, T, H, dv, **f32), dg=torch.empty(B, T, H, dk, **f32),
               dbeta=torch.empty(B, T, H, **f32),
               d_initial_state=torch.empty(N, H, dk, dv, **f32) if want_d_initial_state else None)
    dt = _DTYPES[q.dtype]
    ws_bytes = int(lib.kda_backward_workspace_size(dt, B, T, H, dk, dv, N))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.kda_backward(dt, B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              _ptr(cu_seqlens), N, _ptr(initial_state), _ptr(d_o), _ptr(d_final_state),
                              *(_ptr(out[n]) for n in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")),
                              _ptr(ws), ws_bytes, _stream(dev))
    _raise_if(st)
    return out


def prefill_split_plan(B: int, T: int, H: int, sm_count: int):
    """How ``prefill`` splits B sequences of T tokens and H heads along the sequence on a GPU with
    ``sm_count`` SMs (bf16, d = 128, no cu_seqlens): (segments per sequence, rows per segment,
    workspace bytes); (0, 0, 0) for a single pass. Host arithmetic only (kda_prefill_split_plan)."""
    lib = load()
    P, Ls, nbytes = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _raise_if(lib.kda_prefill_split_plan(int(B), int(T), int(H), int(sm_count), ctypes.byref(P), ctypes.byref(Ls),
                                         ctypes.byref(nbytes)))
    return P.value, Ls.value, nbytes.value


def selftest_wait_timeout(limit_ns: int, device=None):
    """Queue the library's bounded-wait self-test on the current stream of `device`: a kernel
    waits `limit_ns` ns on an mbarrier phase nothing completes and records a time-out in the
    device error word, which the next check_status() raises as KDA_ERR_TIMEOUT."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _raise_if(lib.kda_selftest_wait_timeout(int(limit_ns), _stream(dev)))


def check_status(device=None):
    """Synchronise the current stream and raise KDAError if a kernel flagged an error."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _raise_if(lib.kda_check_status(_stream(dev)))
