"""The C ABI without a GPU: the library builds, loads, exports what include/kda.h declares,
and rejects malformed arguments on the host before touching the device."""

import ctypes
import subprocess

import pytest

import gated_delta_rule_56_gb300 as kda
from gated_delta_rule_56_gb300 import _lib
from gated_delta_rule_56_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return kda.load()


def test_exports_every_declared_symbol(lib):
    names = kda.declared_symbols()
    assert {"kda_prefill", "kda_decode_step", "kda_check_status", "kda_status_string",
            "kda_prefill_workspace_size", "kda_last_error", "kda_version"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", kda.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in exported, f"{n} declared in include/kda.h but not exported"
        assert getattr(lib, n) is not None


def test_status_strings_and_version(lib):
    assert kda.status_string(0) == "KDA_OK"
    assert kda.status_string(1) == "KDA_ERR_INVALID_ARG"
    assert kda.status_string(2) == "KDA_ERR_UNSUPPORTED"
    assert kda.status_string(3) == "KDA_ERR_CUDA"
    assert kda.status_string(4) == "KDA_ERR_TIMEOUT"
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"
    assert kda.version() >= 10000


# cu_seqlens is only compared with NULL by the sizing calls: any non-NULL value marks a packed call.
PACKED = ctypes.c_void_p(16)


def test_workspace_size_is_zero_when_not_split(lib):
    # Many (sequence, head) pairs, fp32 or small heads: one pass, no workspace.
    for f in (lambda *a: lib.kda_prefill_workspace_size(*a), lambda *a: lib.kda_prefill_workspace_size_for(*a, 152)):
        assert f(0, 4, 8192, 32, 128, 128, None, 4) == 0
        assert f(1, 1, 1 << 20, 32, 128, 128, None, 1) == 0    # fp32
        assert f(0, 1, 1 << 20, 32, 64, 64, None, 1) == 0      # d = 64


def test_workspace_size_of_packed_sequences(lib):
    # Packed bf16 sequences (d = 32, 64, 128: all on the tensor-core kernel): 4 bytes per sequence
    # for the longest-first launch order, rounded up to 256; none for one sequence, more than 4096,
    # fp32 or other head sizes.
    for f in (lambda *a: lib.kda_prefill_workspace_size(*a), lambda *a: lib.kda_prefill_workspace_size_for(*a, 152)):
        assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 64) == 256
        assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 100) == 512
        assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 4096) == 4096 * 4
        assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 4097) == 0
        assert f(1, 1, 1 << 20, 32, 128, 128, PACKED, 64) == 0
        assert f(0, 1, 1 << 20, 32, 64, 64, PACKED, 64) == 256
        assert f(0, 1, 1 << 20, 32, 32, 32, PACKED, 64) == 256
        assert f(0, 1, 1 << 20, 32, 96, 96, PACKED, 64) == 0


def test_workspace_size_tells_one_packed_sequence_from_one_unpacked(lib):
    """B = n_seqs = 1: the same sizes mean an unpacked call (split into equal segments on a 152-SM
    GPU: the split plan's size) or a packed one (the packed split planned on the device: the packed
    rows of q~ and the segment states; one packed sequence is planned exactly, into the same P
    segments as the unpacked call; several into at most min(8 n, n + SMs / H))."""
    T, H = 1 << 20, 32
    P, Ls, split = kda.prefill_split_plan(1, T, H, 152)
    assert P == 4 and split > 0
    assert lib.kda_prefill_workspace_size_for(0, 1, T, H, 128, 128, None, 1, 152) == split
    packed = lib.kda_prefill_workspace_size_for(0, 1, T, H, 128, 128, PACKED, 1, 152)
    per_seg = H * 128 * 128 * (4 + 4 + 2)
    assert T * H * 128 * 2 + P * per_seg <= packed < T * H * 128 * 2 + (P + 1) * per_seg
    two = lib.kda_prefill_workspace_size_for(0, 1, T, H, 128, 128, PACKED, 2, 152)
    s_max = min(8 * 2, 2 + 152 // H)  # 6
    assert T * H * 128 * 2 + s_max * per_seg <= two < T * H * 128 * 2 + (s_max + 1) * per_seg
    # On the CPU no device is visible: calls are sized for 0 SMs (no split, no order for one sequence).
    assert lib.kda_prefill_workspace_size(0, 1, T, H, 128, 128, None, 1) == 0
    assert lib.kda_prefill_workspace_size(0, 1, T, H, 128, 128, PACKED, 1) == 0
    assert lib.kda_prefill_workspace_size_for(0, 1, T, H, 128, 128, None, 1, -1) == 0


def test_workspace_size_of_the_packed_split(lib):
    """Packed sequences are split only when there are fewer of them than SMs / H (room for more CTAs
    per head) and at least 4096 rows; otherwise they take the launch order only."""
    f = lambda *a: lib.kda_prefill_workspace_size_for(*a)
    assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 64, 152) == 256          # 64 sequences: order only
    assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 4, 152) == 256          # 152 / 32 = 4 slots: order only
    assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 3, 152) > (1 << 20) * 32 * 256  # 3 < 4 slots: split
    assert f(0, 1, 4095, 32, 128, 128, PACKED, 3, 152) == 256               # too short to split: order
    assert f(0, 1, 1 << 20, 32, 128, 128, PACKED, 3, 64) == 256             # 2 slots on 64 SMs: 3 >= 2
    assert f(1, 1, 1 << 20, 32, 128, 128, PACKED, 3, 152) == 0              # fp32: neither
    assert f(0, 2, 1 << 20, 32, 128, 128, PACKED, 3, 152) == 0              # packed calls have B == 1


def test_debug_dump_rejects_bad_arguments(lib):
    # Sizes and pointers are checked on the host before the device is touched.
    assert lib.kda_prefill_debug_dump(0, 8, 1, *([None] * 8), None, 1, None) == 1
    assert lib.kda_prefill_debug_dump(1, 8, 1, *([None] * 8), None, -1, None) == 1
    assert lib.kda_prefill_debug_dump(1, 8, 1, *([None] * 8), None, 1, None) == 1  # NULL pointers


def test_noalloc_capacity_and_argument_checks(lib):
    assert lib.kda_prefill_noalloc_capacity() == 32 << 20
    # Sizes are checked before the scratch is looked at (no device needed to reject them).
    assert lib.kda_prefill_noalloc(0, -1, 8, 1, 128, 128, *([None] * 6), 1, None, None, None, None) == 1


def test_options_are_checked_before_anything_runs(lib):
    import ctypes
    from gated_delta_rule_56_gb300._lib import KDAOptions
    assert ctypes.sizeof(KDAOptions) == 48  # size_t, float, int, 2 pointers, int (+4 padding), pointer
    null6 = [None] * 6
    for bad in (KDAOptions(0, 0.0, 0), KDAOptions(4, 0.0, 0), KDAOptions(5000, 0.0, 1),
                KDAOptions(16, -1.0, 0), KDAOptions(16, float("nan"), 0), KDAOptions(16, 2e4, 1)):
        assert lib.kda_prefill_ex(0, 1, 64, 1, 128, 128, *null6, 1, None, None, None, ctypes.byref(bad),
                                  None, 0, None) == 1
        assert lib.kda_decode_step_ex(0, 1, 1, 128, 128, *[None] * 7, ctypes.byref(bad), None) == 1
    # State indices need a positive pool size and 4-byte alignment.
    for bad in (KDAOptions(48, 0.0, 0, FAKE, None, 0), KDAOptions(48, 0.0, 0, None, FAKE + 2, 8),
                KDAOptions(48, 0.0, 0, None, None, 0, FAKE + 8)):  # out_gate not 16-byte aligned
        assert lib.kda_prefill_ex(0, 1, 64, 1, 128, 128, *null6, 1, None, None, None, ctypes.byref(bad),
                                  None, 0, None) == 1
    # A caller built against a shorter struct (gate_bound only) is accepted: qk_l2norm defaults to 0,
    # and the call then fails on its NULL tensors, not on the options.
    short = KDAOptions(12, 0.0, 1)
    assert lib.kda_prefill_ex(0, 1, 64, 1, 128, 128, *null6, 1, None, None, None, ctypes.byref(short),
                              None, 0, None) == 1
    assert b"NULL" in lib.kda_last_error()


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced: validation fails first


def _prefill(lib, dtype=0, B=1, T=64, H=2, dk=128, dv=128, ptrs=None, cu=None, n=0, init=None,
             fin=None):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, o=FAKE)
    p.update(ptrs or {})
    return lib.kda_prefill(dtype, B, T, H, dk, dv, p["q"], p["k"], p["v"], p["g"], p["beta"], cu, n,
                           init, p["o"], fin, None, 0, None)


@pytest.mark.parametrize("case,expect", [
    (dict(dtype=7), _lib.KDA_ERR_INVALID_ARG),
    (dict(B=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(dk=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(dk=48, dv=48), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), _lib.KDA_ERR_UNSUPPORTED),
    (dict(ptrs=dict(q=None)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(o=None)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(k=FAKE + 8)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(beta=FAKE + 1)), _lib.KDA_ERR_INVALID_ARG),
    (dict(B=2, cu=FAKE, n=2), _lib.KDA_ERR_INVALID_ARG),
    (dict(cu=FAKE + 2, n=1), _lib.KDA_ERR_INVALID_ARG),
    (dict(cu=FAKE, n=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(init=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),
    (dict(fin=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_arguments_on_host(lib, case, expect):
    st = _prefill(lib, **case)
    assert st == expect, (case, kda.status_string(st), kda.last_error())
    assert kda.last_error() != ""


def _backward(lib, dtype=0, B=1, T=64, H=2, dk=128, dv=128, ptrs=None, cu=None, n=0, init=None, dfin=None,
              dinit=None, ws=FAKE, ws_bytes=None):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, d_o=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, dg=FAKE, dbeta=FAKE)
    p.update(ptrs or {})
    if ws_bytes is None:
        ws_bytes = lib.kda_backward_workspace_size(dtype, B, T, H, 128, 128, n)
    return lib.kda_backward(dtype, B, T, H, dk, dv, p["q"], p["k"], p["v"], p["g"], p["beta"], cu, n, init, p["d_o"],
                            dfin, p["dq"], p["dk"], p["dv"], p["dg"], p["dbeta"], dinit, ws, ws_bytes, None)


@pytest.mark.parametrize("case,expect", [
    (dict(dtype=7), _lib.KDA_ERR_INVALID_ARG),
    (dict(B=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(dk=48, dv=48), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), _lib.KDA_ERR_UNSUPPORTED),
    (dict(B=2, cu=FAKE, n=2), _lib.KDA_ERR_INVALID_ARG),
    (dict(cu=FAKE + 2, n=1), _lib.KDA_ERR_INVALID_ARG),
    (dict(cu=FAKE, n=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(q=None)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(d_o=None)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(dbeta=None)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(dq=FAKE + 8)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(d_o=FAKE + 4)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(beta=FAKE + 1)), _lib.KDA_ERR_INVALID_ARG),
    (dict(dtype=1, ptrs=dict(beta=FAKE + 2)), _lib.KDA_ERR_INVALID_ARG),
    (dict(ptrs=dict(dbeta=FAKE + 2)), _lib.KDA_ERR_INVALID_ARG),
    (dict(init=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),
    (dict(dfin=FAKE + 8), _lib.KDA_ERR_INVALID_ARG),
    (dict(dinit=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),
    (dict(ws=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(ws=FAKE + 8), _lib.KDA_ERR_INVALID_ARG),
    (dict(ws_bytes=1024), _lib.KDA_ERR_INVALID_ARG),
])
def test_backward_rejects_bad_arguments_on_host(lib, case, expect):
    st = _backward(lib, **case)
    assert st == expect, (case, kda.status_string(st), kda.last_error())
    assert kda.last_error() != ""


def test_backward_workspace_sizes(lib):
    """One d x d fp32 state per head and chunk start (16-token chunks for d = 128, 64 for d = 32
    and 64), plus one slot per sequence and a spare."""
    assert lib.kda_backward_workspace_size(0, 4, 8192, 32, 128, 128, 0) == (8192 * 4 // 16 + 4 + 1) * 32 * 128 * 128 * 4
    assert lib.kda_backward_workspace_size(1, 1, 1000, 3, 64, 64, 5) == (1000 // 64 + 5 + 1) * 3 * 64 * 64 * 4
    assert lib.kda_backward_workspace_size(0, 1, 10, 2, 128, 64, 0) == 0  # dk != dv: unsupported


def test_empty_backward_is_a_no_op(lib):
    # No (sequence, head) pair: nothing is queued and no device is needed.
    none = dict(q=None, k=None, v=None, g=None, beta=None, d_o=None, dq=None, dk=None, dv=None, dg=None, dbeta=None)
    assert _backward(lib, B=0, ptrs=none, ws=None, ws_bytes=0) == 0
    assert _backward(lib, H=0, ptrs=none, ws=None, ws_bytes=0) == 0


def test_split_plan_of_the_workloads(lib):
    """On 152 SMs: the B=4 T=8192 H=32 shape (128 pairs) runs as one pass; the 1,048,576-token
    sequence (32 pairs) is cut into 4 segments of 262,144 rows, one CTA per (segment, head)."""
    assert kda.prefill_split_plan(4, 8192, 32, 152) == (0, 0, 0)
    P, Ls, nbytes = kda.prefill_split_plan(1, 1 << 20, 32, 152)
    assert (P, Ls) == (4, 1 << 18)
    # the workspace holds at least the bf16 transition outputs of every row and two fp32 states
    # per (segment, head)
    assert nbytes % 256 == 0 and nbytes >= (1 << 20) * 32 * 128 * 2 + 2 * 4 * 32 * 128 * 128 * 4
    assert kda.prefill_split_plan(1, 1 << 20, 32, 64) == (2, 1 << 19, kda.prefill_split_plan(1, 1 << 20, 32, 64)[2])
    assert kda.prefill_split_plan(1, 4095, 8, 152)[0] == 0  # under two segments of 2048 rows
    assert kda.prefill_split_plan(1, 1 << 20, 32, 0) == (0, 0, 0)  # no SMs: nothing to plan for


@pytest.mark.parametrize("seed", range(4))
def test_split_plan_invariants(lib, seed):
    """Random sizes: P = min(8, SMs / pairs, T / 2048) when that is at least 2 (the rounding of the
    rows to 64 never loses a segment here), segments of a multiple of 64 rows that cover T with
    the last one non-empty, and B P H CTAs that fit one wave."""
    import random
    rnd = random.Random(seed)
    for _ in range(300):
        B, H, sms = rnd.randint(1, 4), rnd.randint(1, 40), rnd.choice([132, 148, 152, 160])
        T = rnd.randint(1, 1 << 21)
        P, Ls, nbytes = kda.prefill_split_plan(B, T, H, sms)
        want = min(8, sms // (B * H), T // 2048)
        if want < 2:
            assert (P, Ls, nbytes) == (0, 0, 0), (B, T, H, sms)
            continue
        assert P == want, (B, T, H, sms, P, want)
        assert Ls % 64 == 0 and (P - 1) * Ls < T <= P * Ls, (B, T, H, P, Ls)
        assert B * P * H <= sms
        assert nbytes % 256 == 0 and nbytes >= B * T * H * 128 * 2


def test_split_plan_rejects_bad_arguments(lib):
    with pytest.raises(kda.KDAError):
        kda.prefill_split_plan(-1, 10, 2, 152)
    with pytest.raises(kda.KDAError):
        kda.prefill_split_plan(1, 10, 2, -5)
    assert lib.kda_prefill_split_plan(1, 10, 2, 152, None, None, None) == _lib.KDA_ERR_INVALID_ARG


def test_empty_prefill_is_a_no_op(lib):
    # No (sequence, head) pair: nothing is queued and no device is needed.
    assert _prefill(lib, B=0, ptrs=dict(q=None, k=None, v=None, g=None, beta=None, o=None)) == 0
    assert _prefill(lib, H=0, T=0, ptrs=dict(q=None, k=None, v=None, g=None, beta=None, o=None)) == 0


@pytest.mark.parametrize("case,expect", [
    (dict(dtype=5), _lib.KDA_ERR_INVALID_ARG),
    (dict(N=-3), _lib.KDA_ERR_INVALID_ARG),
    (dict(dk=96, dv=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(state=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(state=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), _lib.KDA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments_on_host(lib, case, expect):
    a = dict(dtype=0, N=4, H=2, dk=64, dv=64, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, o=FAKE)
    a.update(case)
    st = lib.kda_decode_step(a["dtype"], a["N"], a["H"], a["dk"], a["dv"], a["q"], a["k"], a["v"], a["g"],
                             a["beta"], a["state"], a["o"], None)
    assert st == expect, (case, kda.status_string(st), kda.last_error())


@pytest.mark.parametrize("bound", [0.0, -1.0, float("nan"), 2e4])
def test_gated_entry_points_reject_bad_bound_on_host(lib, bound):
    import ctypes
    st = lib.kda_prefill_gated(0, 1, 4, 1, 128, 128, *([None] * 5), None, 1, None, None, None,
                               ctypes.c_float(bound), None, 0, None)
    assert st == 1 and b"gate_bound" in lib.kda_last_error()
    st = lib.kda_decode_step_gated(0, 1, 1, 128, 128, *([None] * 5), None, None, ctypes.c_float(bound), None)
    assert st == 1 and b"gate_bound" in lib.kda_last_error()


@pytest.mark.parametrize("limit", [0, 10**9 + 1])
def test_selftest_rejects_bad_limit_on_host(lib, limit):
    assert lib.kda_selftest_wait_timeout(limit, None) == 1  # KDA_ERR_INVALID_ARG, nothing launched
    assert b"limit_ns" in lib.kda_last_error()


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 1, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.prefill(x, x, x, x, torch.zeros(1, 4, 1, dtype=torch.bfloat16))
