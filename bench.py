#!/usr/bin/env python3
"""KDA benchmark on GB300: prefill tokens/s (headline), decode tokens/s, roofline fractions.

One step of the headline is one chunked prefill of the workload B=4, T=8192, H=32,
d_k=d_v=128 (bf16 q/k/v/g/beta, fp32 state, zero initial state) through the C ABI. The
decode sub-benchmark runs 1000 consecutive decode steps for 256 sequences x 32 heads x
d=128 from fp32 states ~ N(0, 0.02), with 1000 pre-generated input sets resident on the
device. Inputs are synthetic and seeded (kda_inputs), drawn on the device.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 the script runs under torchrun, one rank per GPU; every rank processes its own
copy of the workload (weak scaling: (sequence, head) pairs are independent, so ranks need
no collective on the data path) and rank 0 prints the line with the max time over ranks.

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the
same workload (there is no other reference implementation of the method).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill tokens/s and decode tokens/s on 1 GB300; % of roofline"
# Backward: algorithmic flops per state element per token (a forward step to rebuild the state:
# decay 1, k-read 2, write 2; the reverse step: decay 1, k-read 2, dq 2, q do^T 2, dS^T k 2, dk 3,
# dSd 2, dg 2, decay 1). Its products run as tf32 tensor-core MMAs, so its roofline is the tf32
# dense rate: the measured bf16 rate times the nominal tf32/bf16 ratio (1.1 / 2.25 PFLOP/s); the
# fp32 FMA rate of the CUDA cores (152 SMs x 128 lanes x 2 flops x 2.07 GHz) is reported beside it.
BWD_FLOPS_PER_ELEM = 22
TF32_PER_BF16 = 1.1 / 2.25
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12

PF = dict(B=4, T=8192, H=32, d=128, chunk=64)
DEC = dict(N=256, H=32, d=128, steps=1000)
NAMES = ("q", "k", "v", "g", "beta")
L2_BYTES = 129 * 2 ** 20


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--decode-steps", type=int, default=DEC["steps"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams the e2e run splits each step's host-to-device copies over")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="leave the varlen and long-context sub-lines out of the default line")
    ap.add_argument("--workload", choices=("varlen", "long", "gated", "l2norm", "outgate", "backward", "fp32", "d64"),
                    default=None,
                    help="time one of the other prefill workloads instead of the headline (one JSON line): "
                         "varlen = 64 packed sequences of U[128, 16384] tokens with initial states; "
                         "long = one sequence of 1,048,576 tokens (B=1, H=32); "
                         "gated = the headline shape with gate logits (decays formed in the kernel); "
                         "l2norm = the headline shape with raw q/k rows L2-normalised in the kernel; "
                         "outgate = the headline shape with the output gate o * sigmoid(z) in the kernel; "
                         "backward = all gradients of the headline shape (kda_backward); "
                         "fp32 = the small fp32 configuration B=1 T=256 H=2 d=64 (tf32 tensor-core kernel); "
                         "d64 = the headline shape with heads of 64 channels (bf16)")
    ap.add_argument("--ncu-case", choices=("prefill", "decode", "decode256", "backward", "long", "varlen", "fp32"),
                    help="run two launches of the small profiling case (for ncu) and exit")
    args = ap.parse_args(argv)
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    # At least 3 untimed warm-up steps whatever is asked; the JSON line reports the count run.
    args.warmup = max(args.warmup, 3)
    return args


# ------------------------------------------------------------------------ ranks ---------

class Ranks:
    """One process per GPU (RANK / LOCAL_RANK / WORLD_SIZE from the launcher). The ranks share
    nothing on the data path (each runs its own copy of the workload); they meet only in the
    barriers around the timed region and in the max over ranks of its duration. NCCL on GPUs;
    `backend="gloo"` with `device="cpu"` runs the same logic on host processes."""

    def __init__(self, gpus, backend=None, device=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world != gpus:
            raise SystemExit(f"--gpus {gpus} but WORLD_SIZE={self.world}")
        self.device = torch.device(device) if device else torch.device("cuda", self.local)
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            if (backend or "nccl") == "nccl":
                dist.init_process_group("nccl", device_id=self.device)
            else:
                dist.init_process_group(backend)
            self.dist = dist
        if self.device.type == "cuda":
            torch.cuda.set_device(self.device)

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if not self.dist:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()

    def job_throughput(self, units_per_rank: float, ms: float) -> float:
        """Whole-job rate: the units every rank processed over the slowest rank's time."""
        return self.world * units_per_rank / (self.max(ms) / 1e3)


# ---------------------------------------------------------------------- clocks ----------

class ClockSampler:
    """nvidia-smi samples (100 ms) of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.ident = None
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            self.ident = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            self.ident = str(device.index)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2], parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i, f in enumerate(r[3]) if f.lower() == "active"})
        top = max(r[0] for r in rows)
        loaded = [r[0] for r in rows if r[0] >= 0.5 * top] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# -------------------------------------------------------------------- roofline ----------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(key, files):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source it was
    taken on is the current one; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(key)
    if not rec or rec.get("source_sha") != source_digest(files):
        return None
    return rec.get("dram_bytes_per_launch")


PREFILL_SOURCES = ["gated_delta_rule_56_gb300/csrc/kda_prefill_tc.cu", "gated_delta_rule_56_gb300/csrc/kda_tc.cuh"]
SPLIT_SOURCES = PREFILL_SOURCES + ["gated_delta_rule_56_gb300/csrc/kda_segmented.cu"]
DECODE_SOURCES = ["gated_delta_rule_56_gb300/csrc/kda_recurrent.cu"]
BACKWARD_SOURCES = ["gated_delta_rule_56_gb300/csrc/kda_backward_chunked.cu"]


def prefill_bytes(B, T, H, d):
    """Algorithmic HBM bytes of one prefill launch: read q, k, v, g (bf16) and beta, write o
    (bf16) -- 1282 B per token-head at d=128 -- plus the fp32 final state per (seq, head)."""
    per_token_head = 4 * d * 2 + 2 + 2 * d
    return B * T * H * per_token_head + B * H * d * d * 4


def decode_bytes(N, H, d):
    """Algorithmic HBM bytes of one decode step: fp32 state read + write per head, bf16
    q, k, g, v and beta read, bf16 o written."""
    return N * H * (2 * d * d * 4 + 4 * d * 2 + 2 + 2 * d)


def existing_files(files):
    return [f for f in files if os.path.exists(os.path.join(ROOT, f))]


# ----------------------------------------------------------------- timing helpers -------

def time_steps(fn, steps, warmup, ranks):
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    ranks.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        fn(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total_ms = ev[0].elapsed_time(ev[steps])
    return total_ms, per


# --------------------------------------------------------------------- our arm ----------

def run_ours(args):
    import gated_delta_rule_56_gb300 as kda
    import kda_inputs as ki
    from gated_delta_rule_56_gb300.build import build

    ranks = Ranks(args.gpus)
    if ranks.local == 0:
        build()
    ranks.barrier()
    kda.load()
    dev = ranks.device
    B, T, H, d = PF["B"], PF["T"], PF["H"], PF["d"]
    x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=ranks.rank)
    o = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
    args_in = [x[n] for n in NAMES]

    def step(_i):
        kda.prefill(*args_in, o=o, final_state=fin)

    step(0)
    kda.check_status()
    peak_bw, peak_tc, peak_kind = measured_peaks()
    with ClockSampler(dev) as clk:
        total_ms, per = time_steps(step, args.steps, args.warmup, ranks)
    kda.check_status()
    tokens = B * T
    value = ranks.job_throughput(tokens * args.steps, total_ms)
    total_ms = ranks.max(total_ms)
    ms = total_ms / args.steps
    kernel_ms = statistics.mean(per)
    alg = prefill_bytes(B, T, H, d)
    achieved = alg / (kernel_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"KDA chunked prefill B={B} T={T} H={H} dk=dv={d} bf16 in, fp32 state, zero init",
                   "global_batch": B * args.gpus, "seq_len": T, "heads": H, "head_dim": d, "chunk": PF["chunk"],
                   "parallelism": f"replicas{args.gpus}" if args.gpus > 1 else "single",
                   "l2": f"no flush: each step reads {alg / 1e9:.2f} GB > {L2_BYTES / 2**20:.0f} MiB L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_bw, "unit": "GB/s",
                     "frac": achieved / peak_bw, "peak_source": peak_kind,
                     "traffic": recorded_traffic("prefill", existing_files(PREFILL_SOURCES)),
                     "alg_bytes_per_launch": alg, "kernel_ms": kernel_ms,
                     "tensor_flop_per_launch": B * T * H * 2 * (1.5 * 64 * d + 64 * d + 3 * d * d),
                     "tensor_frac_of_peak": B * T * H * 2 * (1.5 * 64 * d + 64 * d + 3 * d * d)
                     / (kernel_ms / 1e3) / (peak_tc * 1e12)},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }

    if not args.no_e2e:
        line["e2e"] = run_e2e(args, kda, x, ranks, tokens)
    del x, args_in, o, fin
    torch.cuda.empty_cache()
    if not args.no_decode:
        line["decode"] = run_decode(args, kda, ki, ranks, peak_bw, peak_kind)
    if not args.no_workloads:  # the varlen and long-context workloads, timed the same way
        for w in ("varlen", "long"):
            line[w] = workload_line(args, w, dev, ranks)
    if ranks.rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(ki, dev)
    ranks.close()
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, kda, x, ranks, tokens):
    """Same metric through the public call with host buffers: every step copies that step's
    inputs from pinned host memory to the device and reads o and the final state back, and the
    timed region covers all of it. Steps are pipelined the way a caller streaming work through
    the GPU would: step i's inputs go up (split over --e2e-copy-streams streams) while step i - 1
    computes and step i - 2's results come down (device and host buffers double-buffered, events
    ordering each reuse)."""
    dev = ranks.device
    host = {n: x[n].cpu().pin_memory() for n in NAMES}
    B, T, H, d = PF["B"], PF["T"], PF["H"], PF["d"]
    dev_in = [{n: torch.empty_like(x[n]) for n in NAMES} for _ in range(2)]
    o = [torch.empty(B, T, H, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    fin = [torch.empty(B, H, d, d, dtype=torch.float32, device=dev) for _ in range(2)]
    o_h = [torch.empty(o[0].shape, dtype=o[0].dtype).pin_memory() for _ in range(2)]
    fin_h = [torch.empty(fin[0].shape, dtype=fin[0].dtype).pin_memory() for _ in range(2)]
    s_ups = [torch.cuda.Stream(dev) for _ in range(args.e2e_copy_streams)]
    s_run, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up_done = [[torch.cuda.Event() for _ in s_ups] for _ in range(2)]
    run_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        j = i % 2
        for u, s_up in enumerate(s_ups):  # each upload stream copies one slice of every input
            with torch.cuda.stream(s_up):
                if used[j]:
                    s_up.wait_event(run_done[j])  # the kernel of step i - 2 has read dev_in[j]
                for n in NAMES:
                    src, dst = host[n].view(-1), dev_in[j][n].view(-1)
                    a, b = src.numel() * u // len(s_ups), src.numel() * (u + 1) // len(s_ups)
                    dst[a:b].copy_(src[a:b], non_blocking=True)
                up_done[j][u].record(s_up)
        with torch.cuda.stream(s_run):
            for ev in up_done[j]:
                s_run.wait_event(ev)
            if used[j]:
                s_run.wait_event(down_done[j])    # o[j], fin[j] of step i - 2 are on the host
            kda.prefill(*(dev_in[j][n] for n in NAMES), o=o[j], final_state=fin[j])
            run_done[j].record(s_run)
        with torch.cuda.stream(s_down):
            s_down.wait_event(run_done[j])
            o_h[j].copy_(o[j], non_blocking=True)
            fin_h[j].copy_(fin[j], non_blocking=True)
            down_done[j].record(s_down)
        used[j] = True

    def run(n_steps):
        cur = torch.cuda.current_stream(dev)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(cur)
        for st in (*s_ups, s_run, s_down):
            st.wait_event(start)
        for i in range(n_steps):
            step(i)
        cur.wait_stream(s_down)
        end.record(cur)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    steps = max(3, min(args.e2e_steps, args.steps))
    run(3)  # warm-up
    torch.cuda.synchronize()
    ranks.barrier()
    total_ms = run(steps)
    ranks.barrier()
    kda.check_status()
    value = ranks.job_throughput(tokens * steps, total_ms)
    total_ms = ranks.max(total_ms)
    h2d = sum(host[n].numel() * host[n].element_size() for n in NAMES)
    d2h = o_h[0].numel() * o_h[0].element_size() + fin_h[0].numel() * fin_h[0].element_size()
    return {"value": value, "unit": "tokens/s", "steps": steps,
            "ms_per_step": total_ms / steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "gpu_launches": steps,
            "pipeline": f"upload step i on {len(s_ups)} streams, compute i-1, download i-2"}


def run_decode(args, kda, ki, ranks, peak_bw, peak_kind):
    dev = ranks.device
    N, H, d = DEC["N"], DEC["H"], DEC["d"]
    steps = args.decode_steps
    x = ki.decode_inputs(steps, N, H, d, d, device=dev, seed=100 + ranks.rank)
    state = x["state"]
    o = torch.empty(N, H, d, dtype=torch.bfloat16, device=dev)

    def step(i):
        j = i % steps
        kda.decode_step(x["q"][j], x["k"][j], x["v"][j], x["g"][j], x["beta"][j], state, o=o)

    total_ms, per = time_steps(step, steps, 10, ranks)
    kda.check_status()
    value = ranks.job_throughput(N * steps, total_ms)
    total_ms = ranks.max(total_ms)
    ms = total_ms / steps
    alg = decode_bytes(N, H, d)
    kernel_ms = statistics.mean(per)
    achieved = alg / (kernel_ms / 1e3) / 1e9
    return {"metric": "KDA decode tokens/s (one token for each of N=256 sequences per step, H=32, "
                      "dk=dv=128, bf16 in, fp32 state)",
            "value": value, "unit": "tokens/s", "steps": steps,
            "ms_per_step": ms, "gpu_launches": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_bw, "unit": "GB/s",
                         "frac": achieved / peak_bw, "peak_source": peak_kind,
                         "traffic": recorded_traffic("decode", existing_files(DECODE_SOURCES)),
                         "alg_bytes_per_launch": alg, "kernel_ms": kernel_ms}}


# ----------------------------------------------------------------- CPU baseline ---------

def _oracle_pairs(ki, dev, pairs, tokens):
    """Inputs of `pairs` (batch row, head) problems of `tokens` tokens from the workload's
    seeded inputs, on the host."""
    B, T, H, d = PF["B"], PF["T"], PF["H"], PF["d"]
    x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=0)
    sel = [(i % B, (i * 7) % H) for i in range(pairs)]
    out = []
    for b, h in sel:
        out.append({n: x[n][b:b + 1, :tokens, h:h + 1].cpu() for n in NAMES})
    del x
    return out


def cpu_baseline(ki, dev, pairs=None, tokens=None):
    import oracle
    cores = oracle.max_threads()
    pairs = pairs or max(4 * cores, 32)  # about 20 s of work on the host's cores
    tokens = tokens or PF["T"]
    probs = _oracle_pairs(ki, dev, pairs, tokens)
    # One call over all sampled pairs so OpenMP spreads them over the cores.
    cat = {n: torch.cat([p[n] for p in probs], dim=2) for n in NAMES}
    t0 = time.perf_counter()
    oracle.recurrent(*(cat[n] for n in NAMES), n_threads=cores)
    dt = time.perf_counter() - t0
    token_heads = pairs * tokens
    return {"value": token_heads / PF["H"] / dt, "unit": "tokens/s", "cores": min(cores, pairs),
            "kind": "oracle",
            "sample": f"fp64 recurrence over {pairs} (batch row, head) pairs x {tokens} tokens of the "
                      f"B=4 T=8192 H=32 d=128 workload ({token_heads} token-heads, {dt:.2f} s wall, "
                      f"{dt * min(cores, pairs):.0f} core-seconds); "
                      f"tokens/s = token-heads/s / 32 heads"}


# ------------------------------------------------------------------ reference arm -------

def run_reference(args):
    """The fp64 oracle as the reference arm, on host cores, rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import kda_inputs as ki
    import oracle
    cores = oracle.max_threads()
    pairs, tokens = cores, 256
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))) if torch.cuda.is_available() else "cpu"
    probs = _oracle_pairs(ki, dev, pairs, tokens)
    cat = {n: torch.cat([p[n] for p in probs], dim=2) for n in NAMES}
    for _ in range(args.warmup):
        oracle.recurrent(*(cat[n] for n in NAMES), n_threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrent(*(cat[n] for n in NAMES), n_threads=cores)
    dt = time.perf_counter() - t0
    value = pairs * tokens / PF["H"] * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"KDA chunked prefill B={PF['B']} T={PF['T']} H={PF['H']} dk=dv={PF['d']} "
                                   "bf16 in, fp32 state, zero init"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: fp64 recurrence over {pairs} (batch row, head) pairs x "
                                       f"{tokens} tokens of the workload"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_workload(args):
    """One of the other workloads on its own (one JSON line)."""
    from gated_delta_rule_56_gb300.build import build
    build()
    print(json.dumps(workload_line(args, args.workload, torch.device("cuda", 0), Ranks(1))), flush=True)


def workload_line(args, workload, dev, ranks):
    """The other prefill workloads, timed like the headline: varlen (64 sequences with lengths
    uniform in [128, 16384], seed 0, initial states N(0, 0.02)), long (B=1, T=1,048,576), the
    headline shape with one of the options, or the backward. Returns the workload's line."""
    import gated_delta_rule_56_gb300 as kda
    import kda_inputs as ki
    kda.load()
    H, d = PF["H"], PF["d"]
    if workload == "varlen":
        lengths = ki.varlen_lengths(64, 128, 16384, seed=0)
        x = ki.varlen_inputs(lengths, H, d, d, device=dev, seed=0)
        tokens, n_seq = int(lengths.sum()), int(lengths.numel())
        kw = dict(cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
        alg = tokens * H * (4 * d * 2 + 2 + 2 * d) + 2 * n_seq * H * d * d * 4
        name = f"KDA chunked prefill, varlen: {n_seq} sequences (lengths U[128,16384], seed 0, {tokens} tokens) H={H} dk=dv={d} bf16, fp32 initial states"
    elif workload == "long":
        T = 1 << 20
        x = ki.prefill_inputs(1, T, H, d, d, device=dev, seed=0)
        tokens, n_seq = T, 1
        kw = {}
        alg = prefill_bytes(1, T, H, d)
        name = f"KDA chunked prefill, long context: B=1 T={T} H={H} dk=dv={d} bf16, zero init"
    elif workload == "backward":
        B, T = PF["B"], PF["T"]
        x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=0)
        tokens, n_seq = B * T, B
        kw = dict(d_o=ki.gate_logits_like(x["v"], seed=4))  # dL/do ~ N(0, 1)
        alg = tokens * H * BWD_FLOPS_PER_ELEM * d * d       # algorithmic flops
        name = f"KDA backward (all gradients, fp32 state, tf32 tensor-core products): B={B} T={T} H={H} dk=dv={d} bf16 inputs"
    elif workload == "outgate":
        B, T = PF["B"], PF["T"]
        x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=0)
        tokens, n_seq = B * T, B
        kw = dict(out_gate=ki.gate_logits_like(x["v"], seed=3))  # z ~ N(0, 1): o * sigmoid(z) is stored
        alg = prefill_bytes(B, T, H, d) + tokens * H * d * 2    # + the gate input z (bf16)
        name = f"KDA chunked prefill with the output gate o*sigmoid(z) in the kernel: B={B} T={T} H={H} dk=dv={d} bf16, zero init"
    elif workload == "fp32":
        # the small fp32 configuration: B=1 T=256 H=2 d=64 (the tf32 tensor-core kernel)
        B, T, H, d = 1, 256, 2, 64
        x = ki.prefill_inputs(B, T, H, d, d, dtype=torch.float32, device=dev, seed=0)
        tokens, n_seq = B * T, B
        kw = {}
        alg = tokens * H * (4 * d * 4 + 4 + 4 * d) + n_seq * H * d * d * 4
        name = f"KDA chunked prefill fp32 (tf32 tensor-core kernel): B={B} T={T} H={H} dk=dv={d}, zero init"
    elif workload == "d64":
        B, T, d = PF["B"], PF["T"], 64
        x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=0)
        tokens, n_seq = B * T, B
        kw = {}
        alg = prefill_bytes(B, T, H, d)
        name = f"KDA chunked prefill, heads of 64 channels (the d=128 tensor-core kernel, missing channels zero): B={B} T={T} H={H} dk=dv={d} bf16, zero init"
    elif workload == "l2norm":
        B, T = PF["B"], PF["T"]
        x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=0)
        x["q"], x["k"] = ki.raw_qk_like(x["q"], seed=1), ki.raw_qk_like(x["k"], seed=2)
        tokens, n_seq = B * T, B
        kw = dict(qk_l2norm=True)
        alg = prefill_bytes(B, T, H, d)
        name = f"KDA chunked prefill with q/k L2 normalisation in the kernel: B={B} T={T} H={H} dk=dv={d} bf16, zero init"
    else:
        B, T = PF["B"], PF["T"]
        x = ki.prefill_inputs(B, T, H, d, d, device=dev, seed=0)
        x["g"] = ki.gate_logits_like(x["g"], seed=1)  # logits x; the kernel forms g = -5 sigmoid(x)
        tokens, n_seq = B * T, B
        kw = dict(gate_bound=5.0)
        alg = prefill_bytes(B, T, H, d)
        name = f"KDA chunked prefill with gate logits (g = -5 sigmoid(x) in the kernel): B={B} T={T} H={H} dk=dv={d} bf16, zero init"
    args_in = [x[n] for n in NAMES]
    # A call that the library splits along the sequence (few long sequences; it asks for a
    # workspace) launches 7 kernels: segment bounds, the local pass, the transition pass up to the
    # horizon, the zero test, the transition pass over the rest, the scan and the correction.
    dt_code = 1 if workload == "fp32" else 0  # kda_dtype of the inputs
    split = workload not in ("varlen", "backward") and kda.load().kda_prefill_workspace_size(dt_code, n_seq, tokens // n_seq, H, d, d, None, n_seq) > 0
    launches_per_step = 7 if split else 1
    # Packed sequences with the workspace: the longest-first sort of cu_seqlens, then the prefill.
    if workload == "varlen" and kda.load().kda_prefill_workspace_size(0, 1, tokens, H, d, d, x["cu_seqlens"].data_ptr(), n_seq) > 0:
        launches_per_step = 2
    out = {}
    if workload != "backward":  # outputs allocated once, outside the timed region
        out = dict(o=torch.empty_like(x["v"]),
                   final_state=torch.empty(n_seq, H, d, d, dtype=torch.float32, device=dev))

    def step(_i):
        if workload == "backward":
            kda.backward(*args_in, kw["d_o"])
        else:
            kda.prefill(*args_in, **kw, **out)

    step(0)
    kda.check_status()
    peak_bw, peak_tc, peak_kind = measured_peaks()
    steps, warmup = max(1, min(args.steps, 20)), max(3, min(args.warmup, 5))
    with ClockSampler(dev) as clk:
        total_ms, per = time_steps(step, steps, warmup, ranks)
    kda.check_status()
    kernel_ms = statistics.mean(per)
    achieved = alg / (kernel_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak_bw, "unit": "GB/s", "frac": achieved / peak_bw,
            "peak_source": peak_kind, "alg_bytes_per_launch": alg, "kernel_ms": kernel_ms}
    if workload == "backward":  # tf32 tensor-core products; the fp32 FMA rate beside it
        ach = alg / (kernel_ms / 1e3) / 1e12
        peak_tf32 = peak_tc * TF32_PER_BF16
        roof = {"bound": "tensor", "dtype": "tf32", "achieved": ach, "peak": peak_tf32, "unit": "TFLOP/s",
                "frac": ach / peak_tf32,
                "peak_source": f"{peak_kind} bf16 burst x 1.1/2.25 (nominal dense tf32/bf16)",
                "alg_flops_per_launch": alg, "kernel_ms": kernel_ms,
                "traffic": recorded_traffic("backward", existing_files(BACKWARD_SOURCES)),
                "fp32_alu": {"peak": FP32_ALU_TFLOPS, "frac": ach / FP32_ALU_TFLOPS,
                             "peak_source": "derived from unit counts and the maximum SM clock"}}
        launches_per_step = 1  # d = 128: the chunked kernel writes every output itself (no fills)
    elif workload in ("varlen", "long"):
        roof["traffic"] = recorded_traffic(workload, existing_files(SPLIT_SOURCES if workload == "long" else PREFILL_SOURCES))
    packed = None
    if workload == "long":  # the same tokens as one packed sequence (cu_seqlens = [0, T]): split on the device
        cu = torch.tensor([0, tokens], dtype=torch.int32, device=dev)
        pk_split = kda.load().kda_prefill_workspace_size(0, 1, tokens, H, d, d, cu.data_ptr(), 1) > 0

        def step_packed(_i):
            kda.prefill(*args_in, cu_seqlens=cu, **out)

        step_packed(0)
        kda.check_status()
        pk_total, pk_per = time_steps(step_packed, steps, warmup, ranks)
        kda.check_status()
        pk_ms = statistics.mean(pk_per)
        packed = {"value": ranks.job_throughput(tokens * steps, pk_total), "unit": "tokens/s",
                  "ms_per_step": pk_total / steps, "kernel_ms": pk_ms,
                  "frac": alg / (pk_ms / 1e3) / 1e9 / peak_bw, "split_along_sequence": bool(pk_split),
                  "gpu_launches": steps * (8 if pk_split else 1),
                  "how": "cu_seqlens = [0, T]: the segments are planned on the device (planner, local pass, "
                         "transition pass to the horizon, zero test, rerun, scan, correction)"}
    del x, args_in, kw, out
    torch.cuda.empty_cache()
    line = {
        "metric": f"KDA {'backward' if workload == 'backward' else 'prefill'} tokens/s ({workload})",
        "value": ranks.job_throughput(tokens * steps, total_ms), "unit": "tokens/s",
        "n_gpus": ranks.world, "steps": steps, "warmup": warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
        "dtype": "tf32" if workload == "fp32" else "bf16", "data": "synthetic",
        "config": {"workload": name, "pairs": n_seq * H, "split_along_sequence": bool(split)},
        "roofline": roof,
        "gpu_launches": steps * launches_per_step, "clocks": clk.summary()}
    if packed:
        line["packed"] = packed
    return line


def ncu_case(kind):
    """Small cases sized for an ncu capture: inputs larger than L2, a few GB on the device at
    most. prefill: B=4 T=2048 H=32 d=128 (128 CTAs); decode: N=64 H=32 d=128 (2048 CTAs);
    decode256: the decode workload's own step, N=256 H=32 d=128 (a 537 MB state, past L2);
    backward: B=2 T=1024 H=32 d=128 (512 CTAs); long: B=1 T=65,536 H=32 d=128, split along the
    sequence like the long-context workload (its first prefill launch is the local pass); varlen:
    the first 8 sequences of the varlen workload's lengths, H=32; fp32: fp32 inputs, B=4 T=2048
    H=32 d=64 (the tf32 tensor-core kernel, 128 CTAs of 32 chunks)."""
    import gated_delta_rule_56_gb300 as kda
    import kda_inputs as ki
    from gated_delta_rule_56_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    if kind == "prefill":
        x = ki.prefill_inputs(4, 2048, 32, 128, 128, device=dev, seed=0)
        for _ in range(2):
            o, _s = kda.prefill(*(x[n] for n in NAMES))
    elif kind == "long":
        x = ki.prefill_inputs(1, 1 << 16, 32, 128, 128, device=dev, seed=0)
        for _ in range(2):
            o, _s = kda.prefill(*(x[n] for n in NAMES))
    elif kind == "varlen":
        lengths = ki.varlen_lengths(64, 128, 16384, seed=0)[:8]
        x = ki.varlen_inputs(lengths, 32, 128, 128, device=dev, seed=0)
        for _ in range(2):
            o, _s = kda.prefill(*(x[n] for n in NAMES), cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    elif kind == "decode256":
        x = ki.decode_inputs(2, 256, 32, 128, 128, device=dev, seed=0)
        st = x["state"].clone()
        for t in range(2):
            o = kda.decode_step(*(x[n][t] for n in NAMES), st)
    elif kind == "fp32":
        x = ki.prefill_inputs(4, 2048, 32, 64, 64, dtype=torch.float32, device=dev, seed=0)
        for _ in range(2):
            o, _s = kda.prefill(*(x[n] for n in NAMES))
    elif kind == "backward":
        x = ki.prefill_inputs(2, 1024, 32, 128, 128, device=dev, seed=0)
        do = ki.gate_logits_like(x["v"], seed=4)
        for _ in range(2):
            o = kda.backward(*(x[n] for n in NAMES), do)["dq"]
    else:
        x = ki.decode_inputs(2, 64, 32, 128, 128, device=dev, seed=0)
        st = x["state"].clone()
        for t in range(2):
            o = kda.decode_step(*(x[n][t] for n in NAMES), st)
    kda.check_status()
    print(json.dumps({"ncu_case": kind, "checksum": float(o.float().abs().mean())}))


def main():
    args = parse()
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    if args.workload:
        run_workload(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
