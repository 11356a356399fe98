#!/usr/bin/env python3
"""Benchmark of the MDN memory update on one GB300 (or N replicas).

Main metric: chunkwise-forward tokens/s on the largest prefill workload, the
variable-length packed batch (32768 tokens in sequences of 128..4096 tokens,
H=16, d=128, bf16 q/k/v, fp32 gates and states), with the roofline of its
dominant kernel and of the whole call.  The other prefill workloads (the
400M- and 1.3B-model-shaped batches, the tiny fp32 case) follow under
``other_workloads`` with the same keys; the decode step (256 sequences x 16
heads x d=128, 1000 steps) is reported in ``decode``.

Algorithmic work (what the method itself must move and compute, per token
and head, d = dk = dv, C = 64): 12 d^2 + 8 C d + 4 C d + C^2 / 3 FLOP; HBM
bytes: q, k, v read and o written (4 d elements), the gates (3 or 4 fp32),
plus per (sequence, head) the initial states read (when given) and the final
states written (2 d^2 fp32 each).  The prepared blocks the two kernels pass
through HBM are an intermediate of this implementation, reported as such,
never as algorithmic bytes.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Timing: W warm-up steps, then exactly K steps; before every timed step L2 is
flushed by writing a 256 MiB buffer and then reading a second one (outside
the timed interval, so the flush's own dirty lines are written back before
the timer starts); each step is bracketed by CUDA events on the launching
stream, and the library records caller-created events at its stage
boundaries so the dominant kernel is timed live.  With N > 1 (torchrun) every rank runs the same workload independently
(replicas: the method has no exchange step), timing is bracketed by a barrier
and synchronize on both sides and the MAX over ranks is taken.
"""
import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
SMS = 152
FP32_LANES_PER_SM = 128          # FFMA lanes per SM per clock
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["mdn", "reference"], default="mdn")
    p.add_argument("--workload", default=W.VARLEN_PACKED.name,
                   choices=[n for n, w in W.BY_NAME.items() if not w.decode_steps])
    p.add_argument("--decode-steps", type=int, default=W.DECODE.decode_steps)
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-vres", action="store_true",
                   help="skip timing the forward that also writes the residuals")
    p.add_argument("--no-inputs", action="store_true",
                   help="skip timing the gate / query-key preparation kernel")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-backward", action="store_true",
                   help="skip timing the gradient pass")
    p.add_argument("--no-block", action="store_true",
                   help="skip timing the token-mixer block")
    p.add_argument("--no-other-workloads", action="store_true",
                   help="skip timing the other prefill workloads")
    p.add_argument("--decode-only", action="store_true",
                   help="time only the decode workload and print its object")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="minimum CPU time of the oracle baseline sample")
    return p.parse_args()


# ---------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = list(csv.reader(io.StringIO(f.read())))
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_record(kernel_key, workload, source_file):
    """Per-launch DRAM bytes of one kernel on one workload from a committed
    ncu summary, if it was taken on the current source of the kernel (sha256
    of its .cu file)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get("%s|%s" % (kernel_key, workload))
        with open(source_file, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except (OSError, ValueError, AttributeError):
        return None
    if not rec or rec.get("source_sha256") != sha:
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------- work units

def path_flops_per_token_head(d, C=64):
    """The method's algorithmic FLOPs per (token, head) for the whole chunk
    forward: state products 12 d^2 (K and Q against [S | M], the carry),
    Grams and the Y, Z rows 8 C d, U and the intra-chunk output 4 C d, the
    triangular solve C^2 / 3."""
    return 12 * d * d + 8 * C * d + 4 * C * d + C * C // 3


def kernel_flops_per_token_head(d, C=64):
    """FLOPs each kernel of this implementation performs per (token, head):
    the state pass the state products and [T; A_O T] R (12 d^2 + 4 C d), the
    prep the two Grams, A_O T and the triangular inverse."""
    return {"prep": 4 * C * d + 2 * C * C + C * C // 3,
            "state": 12 * d * d + 4 * C * d}


PREP_BLOCK_BYTES = {"bf16": 18432, "fp32": 34816}   # bf16 operands / split hi-lo operands


def io_bytes(x):
    """Algorithmic HBM bytes, split by what reads or writes them."""
    el = 2 if x["dtype"] == "bf16" else 4
    th = sum(seq_lengths(x)) * x["H"]
    D = x["D"]
    n_gates = 3 + (1 if x["beta"] is not None else 0)
    n_chain = x["n_seq"] * x["H"]
    state = n_chain * D * D * 4
    return {"qk": th * 2 * D * el, "v": th * D * el, "o": th * D * el,
            "gates": th * n_gates * 4,
            "states_in": 2 * state if x["S0"] is not None else 0,
            "states_out": 2 * state}


def intermediate_bytes(x, tensor=True):
    """Prepared blocks written by the prep kernel and read by the state pass,
    and for fp32 inputs the hi / lo bf16 parts of q, k, v (intermediates of
    this implementation, not algorithmic work)."""
    chunks = sum((L + 63) // 64 for L in seq_lengths(x)) * x["H"]
    blocks = PREP_BLOCK_BYTES[x["dtype"]] * chunks
    if x["dtype"] == "fp32":
        blocks += 2 * 3 * 2 * sum(seq_lengths(x)) * x["H"] * x["D"]   # written, then read
    return blocks


def algorithmic(x, what):
    """(bytes, flops) of the whole path ("call") or of one kernel."""
    b = io_bytes(x)
    th = sum(seq_lengths(x)) * x["H"]
    if what == "call":
        return (sum(b.values()), path_flops_per_token_head(x["D"]) * th)
    fl = kernel_flops_per_token_head(x["D"])[what] * th
    if what == "prep":
        return b["qk"] + b["gates"], fl
    return b["qk"] + b["v"] + b["o"] + b["states_in"] + b["states_out"], fl


def roofline_of(x, what, tensor, ms, peaks, peak_src):
    """Binding roofline of the whole call or one kernel: whichever of its
    algorithmic HBM bytes or FLOPs needs more time at the measured peak.
    bf16 inputs: the bf16 tensor peak.  fp32 inputs: the state pass's
    contractions are three bf16 products each (split operands), so its peak
    is a third of the bf16 one; the fp32 prep's inverse and A_O T run on the
    CUDA cores around its tcgen05 Grams, so it is held to the FFMA peak."""
    by, fl = algorithmic(x, what)
    s = ms / 1e3
    fp32 = x["dtype"] == "fp32"
    if fp32 and what == "prep":
        tensor = False
    if tensor and fp32:
        tflops_peak = peaks["bf16_tflops"] / 3.0
        fl_src = "%s bf16 burst / 3 (split operands: three bf16 products per fp32 one)" % peak_src
    elif tensor:
        tflops_peak = peaks["bf16_tflops"]
        fl_src = "%s bf16 burst" % peak_src
    else:
        tflops_peak = SMS * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        fl_src = "fp32 FFMA from unit counts (152 SMs x 128 lanes x 2 x max clock)"
    t_fl = fl / (tflops_peak * 1e12)
    t_by = by / (peaks["hbm_gbs"] * 1e9)
    common = {"algorithmic_bytes": by, "algorithmic_flops": fl, "ms": ms}
    if t_by >= t_fl:
        ach = by / s / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": ach / peaks["hbm_gbs"], "peak_source": "%s HBM copy" % peak_src,
             "other_roof_frac": (fl / s / 1e12) / tflops_peak}
    else:
        ach = fl / s / 1e12
        r = {"bound": "tensor" if tensor else "alu", "achieved": ach, "peak": tflops_peak,
             "unit": "TFLOP/s", "frac": ach / tflops_peak, "peak_source": fl_src,
             "other_roof_frac": (by / s / 1e9) / peaks["hbm_gbs"]}
    r.update(common)
    return r


def seq_lengths(x):
    if x["cu_seqlens"] is not None:
        cu = x["cu_seqlens"].tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    return [x["T"]] * x["B"]


# ---------------------------------------------------------------- arms

def run_cpu_oracle(x, seconds, max_seqs=None):
    """Time the fp64 oracle (as it stands) on the host cores."""
    from oracle import recurrence
    import numpy as np
    lens = seq_lengths(x)
    n_use = len(lens) if max_seqs is None else min(max_seqs, len(lens))
    cu = [0]
    for L in lens[:n_use]:
        cu.append(cu[-1] + L)
    H, D = x["H"], x["D"]
    T_use = cu[-1]
    sl = slice(0, T_use)
    flat = lambda t: t.reshape(-1, *t.shape[2:])[sl].double().numpy()
    args = [flat(x[n]) for n in ("q", "k", "v", "alpha", "mu", "eta")]
    beta = flat(x["beta"]) if x["beta"] is not None else None
    S0 = x["S0"][:n_use].double().numpy() if x["S0"] is not None else None
    M0 = x["M0"][:n_use].double().numpy() if x["M0"] is not None else None
    cores = host_cores()
    reps, t0 = 0, time.perf_counter()
    while True:
        recurrence.forward(*args, beta=beta, S0=S0, M0=M0,
                           cu_seqlens=np.array(cu, np.int32), n_threads=cores)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    tokens = T_use * reps
    return {"value": tokens / dt, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d of %d sequences (%d tokens x %d heads, d=%d), fp64 "
                      "token recurrence, %d repetition(s) in %.1f s" %
                      (n_use, len(lens), T_use, H, D, reps, dt)}


def reference_arm(args, rank, world):
    """The oracle timed on the host cores, same metric/config as the GPU arm."""
    if rank != 0:
        return
    w = W.BY_NAME[args.workload]
    x = W.make_prefill(w)
    steps, warm = args.steps, args.warmup
    # each step: a bounded sample (two sequences) so the run ends in minutes
    per = []
    for i in range(warm + steps):
        r = run_cpu_oracle(x, seconds=0.0, max_seqs=2)
        if i >= warm:
            per.append(r)
    val = statistics.mean(r["value"] for r in per)
    tokens_per_step = sum(seq_lengths(x)[:2])
    line = {
        "impl": "reference", "metric": "MDN chunkwise fwd tokens/s",
        "value": val, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": 1e3 * tokens_per_step / val,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_of(w, x, "none (host oracle)"),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": per[0]["cores"],
                         "kind": "oracle", "sample": per[0]["sample"] + " per step"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, x, l2):
    cfg = {"workload": w.name, "B": x["B"], "T": x["T"], "H": x["H"],
           "d_k": x["D"], "d_v": x["D"], "chunk": 64, "inputs": x["dtype"],
           "gates_states": "fp32", "n_seq": x["n_seq"], "l2": l2,
           "parallelism": "replicas"}
    return cfg


class L2Flush:
    """Empties L2 of every input before a timed step: writes a buffer larger
    than L2, then reads a second one, so that the timed kernels start with
    neither cached inputs nor the write flush's dirty lines still waiting to
    be written back (those would otherwise go out to HBM during the timed
    kernels and be charged to them)."""

    def __init__(self, nbytes, dev):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


def time_prefill(mdn, x_dev, w, steps, warmup, world, flush):
    dev = x_dev["q"].device
    o = torch.empty_like(x_dev["v"])
    S_T = torch.empty((x_dev["n_seq"], x_dev["H"], x_dev["D"], x_dev["D"]),
                      dtype=torch.float32, device=dev)
    M_T = torch.empty_like(S_T)
    need = mdn.workspace_size(x_dev["n_seq"], x_dev["B"] * x_dev["T"], x_dev["H"],
                              x_dev["D"], x_dev["q"].dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    info = {}

    def step(evs=None):
        mdn.chunk_fwd(x_dev["q"], x_dev["k"], x_dev["v"], x_dev["alpha"],
                      x_dev["mu"], x_dev["eta"], x_dev["beta"], x_dev["S0"],
                      x_dev["M0"], cu_seqlens=x_dev["cu_seqlens"], o=o, S_T=S_T,
                      M_T=M_T, workspace=ws, stage_events=evs, info=info)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    # Timed steps: events around the whole call only, so the state pass may
    # overlap the prep kernel's last wave (programmatic dependent launch).
    cur = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(cur)
        step()
        evs[i][1].record(cur)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    st = mdn.device_status()
    if st != 0:
        raise RuntimeError("device status %d after the timed region" % st)
    total = [a.elapsed_time(b) for a, b in evs]
    # Per-stage split from separate steps with an event between the kernels
    # (which serialises them): for the per-kernel rooflines only.
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        step(sevs[i])
    torch.cuda.synchronize()
    stage0 = [e[0].elapsed_time(e[1]) for e in sevs]
    stage1 = [e[1].elapsed_time(e[2]) for e in sevs]
    return {"total_ms": sum(total), "stage_ms": [statistics.mean(stage0),
                                                 statistics.mean(stage1)],
            "wall_s": wall, "path": info.get("path"),
            "launches_per_step": mdn.chunk_fwd_kernel_count(
                x_dev["n_seq"], x_dev["B"], x_dev["T"], x_dev["H"], x_dev["D"], x_dev["q"].dtype,
                x_dev["cu_seqlens"] is not None)}


def time_vres(mdn, x_dev, steps, warmup, flush):
    """The forward that also writes every token's residual (mdn_chunk_fwd_vres),
    same inputs, L2 flushed before each step: ms per step."""
    dev = x_dev["q"].device
    vres = torch.empty_like(x_dev["v"])
    o = torch.empty_like(x_dev["v"])

    def step():
        mdn.chunk_fwd(x_dev["q"], x_dev["k"], x_dev["v"], x_dev["alpha"], x_dev["mu"],
                      x_dev["eta"], x_dev["beta"], x_dev["S0"], x_dev["M0"],
                      cu_seqlens=x_dev["cu_seqlens"], o=o, vres=vres)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        step()
        b.record(cur)
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ts), vres.numel() * vres.element_size()


GATE_PARAMS = dict(a=1.0, b=0.0, s=1.0, tau=8.0, log_mu_min=-2.0, comba_d=0.0)


def time_inputs(mdn, x_dev, steps, warmup, flush, peaks):
    """mdn_prepare_inputs on the workload's q, k with synthetic projections
    z ~ N(0, 1): ms per call and its HBM roofline (reads q, k and four
    projections, writes q_hat, k_hat and four gates)."""
    q, k = x_dev["q"], x_dev["k"]
    g = torch.Generator(device=q.device).manual_seed(7)
    z = [torch.randn(q.shape[:-1], generator=g, device=q.device) for _ in range(4)]
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    for _ in range(warmup):
        flush.zero_()
        mdn.prepare_inputs(q, k, *z, q_out=qo, k_out=ko, **GATE_PARAMS)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(q.device)
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        mdn.prepare_inputs(q, k, *z, q_out=qo, k_out=ko, **GATE_PARAMS)
        b.record(cur)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ts)
    rows = q.numel() // q.shape[-1]
    nbytes = 4 * q.numel() * q.element_size() + rows * 8 * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"what": "gates from their projections + L2-normalised q, k (mdn_prepare_inputs)",
            "ms_per_call": ms, "rows": rows,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "algorithmic_bytes": nbytes}}


def bwd_flops_per_token_head(d, C=64):
    """FLOPs the gradient pass performs per (token, head): the state products
    of the chunk kernel (P S0, P M0, Q S0, Q M0, Kh dS, Kh dM and the three
    n x dk accumulators, 24 d^2), the reverse chain (WS dS, WM dM and the two
    state-adjoint updates, 12 d^2), and the chunk-local products (Grams, T R,
    dO Vres^T, dR Vres^T, A^T dO, T^T dVres and the four C x C by C x d
    products, 14 C d), plus the triangular inverse (C^2 / 3)."""
    return 36 * d * d + 14 * C * d + C * C // 3


def bwd_bytes(x):
    """Algorithmic HBM bytes of one gradient pass: q, k, v and dO read, dq,
    dk, dv written (input dtype); the four gates read and their gradients
    written (fp32); every chunk's entry states read (the saved data, in the
    input dtype); the final-state adjoints read and dS0, dM0 written
    (fp32)."""
    lens = seq_lengths(x)
    th = sum(lens) * x["H"]
    D = x["D"]
    el = 4 if x["dtype"] == "fp32" else 2
    chunks = sum((n + 63) // 64 for n in lens) * x["H"]
    seq_heads = len(lens) * x["H"]
    return (7 * th * D * el + 8 * th * 4 + chunks * 2 * D * D * el +
            seq_heads * 4 * D * D * 4)


def time_backward(mdn, x, x_dev, steps, warmup, flush, peaks):
    """mdn_chunk_bwd on the workload (its forward's chunk entry states taken
    once beforehand, random adjoints of o and of the final states), L2
    flushed before every timed call: ms per call, tokens/s, and the roofline
    of the whole pass: whichever of its algorithmic bytes (HBM) or FLOPs
    (bf16 tensor peak: the bf16 pass runs its products on tcgen05; fp32
    inputs take the CUDA-core kernels, FFMA peak) needs more time.  Also
    the forward that saves those states (mdn_chunk_fwd_states), timed the
    same way, the gradient pass that also reuses that forward's T and A_O T
    (its workspace kept), and the training step those two make (each timed
    after an L2 flush, as a layer's backward runs long after its forward)."""
    d = x_dev
    _, _, _, Sc, Mc = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                                    d["beta"], d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"],
                                    return_chunk_states=True)
    fws = torch.empty(max(256, mdn.workspace_size(d["n_seq"], d["B"] * d["T"], d["H"], d["D"],
                                                  d["q"].dtype)),
                      dtype=torch.uint8, device=d["q"].device)

    def fwd_call():
        return mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], d["beta"],
                             d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"], workspace=fws,
                             S_chunks=Sc, M_chunks=Mc)
    g = torch.Generator(device=d["q"].device).manual_seed(11)
    do = torch.randn(d["v"].shape, generator=g, device=d["v"].device).to(d["v"].dtype)
    n_seq, H, D = d["n_seq"], d["H"], d["D"]
    dS = torch.randn((n_seq, H, D, D), generator=g, device=do.device) * 0.1
    dM = torch.randn((n_seq, H, D, D), generator=g, device=do.device) * 0.1
    need = mdn.chunk_bwd_workspace_size(n_seq, d["B"] * d["T"], H, D, d["q"].dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=do.device)

    bf16_in = d["q"].dtype == torch.bfloat16

    def call():
        return mdn.chunk_bwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], Sc, Mc,
                             do, beta=d["beta"], dS_T=dS, dM_T=dM, cu_seqlens=d["cu_seqlens"],
                             workspace=ws)

    def call_reuse():
        return mdn.chunk_bwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], Sc, Mc,
                             do, beta=d["beta"], dS_T=dS, dM_T=dM, cu_seqlens=d["cu_seqlens"],
                             workspace=ws, fwd_workspace=fws)

    def timed(fn):
        for _ in range(warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream(do.device)
        ts = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            fn()
            b.record(cur)
            ts.append((a, b))
        torch.cuda.synchronize()
        st = mdn.device_status()
        if st != 0:
            raise RuntimeError("device status %d after the gradient pass" % st)
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    fwd_ms = timed(fwd_call)
    ms = timed(call)
    reuse_ms = timed(call_reuse) if bf16_in else ms
    tokens = sum(seq_lengths(x))
    fl = bwd_flops_per_token_head(D) * tokens * H
    by = bwd_bytes(x)
    s = ms / 1e3
    bf16 = x["dtype"] != "fp32"
    if bf16:
        fpeak, fsrc, fbound = peaks["bf16_tflops"], "measured bf16 burst", "tensor"
    else:
        fpeak = SMS * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        fsrc, fbound = "fp32 FFMA from unit counts (152 SMs x 128 lanes x 2 x max clock)", "alu"
    f_fl = fl / s / 1e12 / fpeak
    f_by = by / s / 1e9 / peaks["hbm_gbs"]
    if f_by >= f_fl:
        roof = {"bound": "hbm", "achieved": by / s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": f_by, "peak_source": "measured HBM copy", "other_roof_frac": f_fl}
    else:
        roof = {"bound": fbound, "achieved": fl / s / 1e12, "peak": fpeak, "unit": "TFLOP/s",
                "frac": f_fl, "peak_source": fsrc, "other_roof_frac": f_by}
    roof.update({"algorithmic_bytes": by, "algorithmic_flops": fl})
    launches = (5 if bf16 else 3) + (1 if d["cu_seqlens"] is not None else 0)
    return {"what": "gradient pass (mdn_chunk_bwd) from the forward's chunk entry states",
            "ms_per_call": ms, "tokens_per_s": tokens / s,
            "forward_with_states_ms": fwd_ms,
            "ms_per_call_reusing_forward_workspace": reuse_ms,
            "training_step": {"what": "mdn_chunk_fwd_states + mdn_chunk_bwd reusing its T, A_O T",
                              "ms": fwd_ms + reuse_ms,
                              "tokens_per_s": tokens / ((fwd_ms + reuse_ms) / 1e3)},
            "ratio_to_forward": None, "gpu_launches_per_call": launches,
            "kernels": ("chunk_prep_tc (the forward's), bwd_vec, bwd_chain_tc, bwd_chunk_tc, "
                        "bwd_gates" if bf16 else "bwd_prep, bwd_chain, bwd_chunk"),
            "roofline": roof}


def time_block(mdn, x_dev, steps, warmup, flush):
    """mdn_block_fwd (the token-mixer block around the core) on the
    workload's token layout with d_model = H d and seeded random weights:
    ms per call and tokens/s."""
    d = x_dev
    dev = d["q"].device
    H, D = d["H"], d["D"]
    dm = H * D
    g = torch.Generator(device=dev).manual_seed(13)
    dt = d["q"].dtype
    T_total = d["B"] * d["T"]
    B, T = (1, T_total) if d["cu_seqlens"] is not None else (d["B"], d["T"])
    xb = torch.randn((B, T, dm), generator=g, device=dev).to(dt)
    W_in = (torch.randn((dm, 4 * H * D + 4 * H), generator=g, device=dev) / dm ** 0.5).to(dt)
    conv_w = torch.randn((3 * H * D, 4), generator=g, device=dev) * 0.5
    rms_w = torch.ones(D, device=dev)
    W_o = (torch.randn((H * D, dm), generator=g, device=dev) / dm ** 0.5).to(dt)
    need = mdn.block_fwd_workspace_size(d["n_seq"], T_total, H, D, dm, dt)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def call():
        mdn.block_fwd(xb, W_in, conv_w, rms_w, W_o, H, D, cu_seqlens=d["cu_seqlens"],
                      workspace=ws, **GATE_PARAMS)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        call()
        b.record(cur)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ts)
    gemm_flops = 2 * T_total * dm * (4 * H * D + 4 * H) + 2 * T_total * H * D * dm
    return {"what": "token-mixer block (mdn_block_fwd): projection GEMM, short convolution, "
                    "gates and q/k, MDN core, RMSNorm and output gate, output GEMM",
            "d_model": dm, "ms_per_call": ms, "tokens_per_s": T_total / (ms / 1e3),
            "projection_flops": gemm_flops,
            "weights": "seeded random (no trained weights are needed to time the block)"}


def time_e2e(mdn, x, x_dev, steps, warmup):
    """Same metric through the public API from pinned host buffers: every
    step copies its inputs host->device, runs, and copies o and the final
    states back to pinned host memory.  Steps stream as a user would run
    them: host->device copies, kernels and device->host copies on three
    streams over two device buffer sets, so step i's copies overlap the
    kernels of its neighbours.  Time = first copy in to last copy out, / K."""
    names = ["q", "k", "v", "alpha", "mu", "eta", "beta", "S0", "M0"]
    host = {n: x[n].pin_memory() for n in names if x[n] is not None}
    o_h = torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory()
    S_h = torch.empty((x["n_seq"], x["H"], x["D"], x["D"])).pin_memory()
    M_h = torch.empty_like(S_h).pin_memory()
    devc = x_dev["q"].device
    need = mdn.workspace_size(x["n_seq"], x["B"] * x["T"], x["H"], x["D"], x["q"].dtype)
    bufs = []
    for _ in range(2):
        bufs.append({
            "in": {n: torch.empty_like(x_dev[n]) for n in host},
            "o": torch.empty_like(x_dev["v"]),
            "S": torch.empty((x["n_seq"], x["H"], x["D"], x["D"]), device=devc),
            "M": torch.empty((x["n_seq"], x["H"], x["D"], x["D"]), device=devc),
            "ws": torch.empty(need, dtype=torch.uint8, device=devc),
        })
    cu = x_dev["cu_seqlens"]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in (o_h, S_h, M_h))
    s_in, s_run, s_out = (torch.cuda.Stream(devc) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "run", "out")}
    for k in ev:               # every buffer starts free
        for e in ev[k]:
            e.record(torch.cuda.current_stream(devc))

    def step(i):
        b = bufs[i & 1]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["run"][i & 1])        # inputs of step i-2 consumed
            for n, t in host.items():
                b["in"][n].copy_(t, non_blocking=True)
            ev["in"][i & 1].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev["in"][i & 1])
            s_run.wait_event(ev["out"][i & 1])       # outputs of step i-2 copied out
            d = b["in"]
            mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                          d.get("beta"), d.get("S0"), d.get("M0"), cu_seqlens=cu,
                          o=b["o"], S_T=b["S"], M_T=b["M"], workspace=b["ws"],
                          stream=s_run)
            ev["run"][i & 1].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["run"][i & 1])
            o_h.copy_(b["o"], non_blocking=True)
            S_h.copy_(b["S"], non_blocking=True)
            M_h.copy_(b["M"], non_blocking=True)
            ev["out"][i & 1].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_run)
    t1.record(s_out)
    t1.synchronize()             # the last result is on the host now
    return t0.elapsed_time(t1) / steps, h2d, d2h


def time_decode(mdn, steps, dev, peaks):
    w = W.DECODE
    S0, M0 = W.make_decode_state(w, device=dev)
    xs = W.make_decode_steps(w, steps, device=dev)
    o = torch.empty_like(xs["v"][0])
    S, M = S0.clone(), M0.clone()
    for t in range(3):                        # warm-up on a scratch copy
        mdn.decode_step(xs["q"][t], xs["k"][t], xs["v"][t], xs["alpha"][t],
                        xs["mu"][t], xs["eta"][t], S, M, o=o)
    S.copy_(S0)
    M.copy_(M0)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for t in range(steps):
        mdn.decode_step(xs["q"][t], xs["k"][t], xs["v"][t], xs["alpha"][t],
                        xs["mu"][t], xs["eta"][t], S, M, o=o)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    st = mdn.device_status()
    if st != 0:
        raise RuntimeError("device status %d after decode" % st)
    N, H, D = w.B, w.H, w.D
    bytes_step = (N * H * D * D * 4 * 4            # S, M read + write
                  + N * H * D * 2 * 4              # q, k, v read, o write (bf16)
                  + N * H * 4 * 3)                 # gates
    per_step_s = ms / 1e3 / steps
    achieved = bytes_step / per_step_s / 1e9
    return {"metric": "MDN decode steps/s", "value": steps / (ms / 1e3),
            "unit": "steps/s", "tokens_per_s": N * steps / (ms / 1e3),
            "steps": steps, "ms_per_step": ms / steps,
            "config": {"workload": w.name, "N": N, "H": H, "d_k": D, "d_v": D,
                       "inputs": "bf16", "states": "fp32, in place",
                       "l2": "states (1.07 GB) exceed L2; no flush"},
            "gpu_launches": steps,
            "roofline": {"bound": "hbm", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": traffic_record("decode_step", w.name, os.path.join(
                             ROOT, "momentum_delta_rule_gb300", "csrc", "mdn_decode.cu"))}}


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(val, world, dev):
    if world == 1:
        return val
    import torch.distributed as dist
    t = torch.tensor([val], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank, max_ms, steps, world):
    """Tokens per second of the whole job: every rank processes its own
    replica of `tokens_per_rank` tokens per step, and the slowest rank's time
    (`max_ms` over `steps` steps) bounds the job."""
    return world * tokens_per_rank / (max_ms / steps / 1e3)


KERNEL_SOURCES = {"chunk_prep_tc": "mdn_prep_tc.cu", "chunk_state_tc": "mdn_chunk_tc.cu",
                  "chunk_prep_split": "mdn_chunk_simt.cu"}


def measure_prefill(mdn, w, x, dev, args, steps, warmup, world, flush, peaks, peak_src,
                    e2e=True):
    """Device-timed chunk forward of one workload with its rooflines (the
    dominant kernel's and the whole call's) and, optionally, the same metric
    end to end from pinned host buffers."""
    x_dev = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    r = time_prefill(mdn, x_dev, w, steps, warmup, world, flush)
    max_ms = max_over_ranks(r["total_ms"], world, dev)
    tokens = sum(seq_lengths(x))
    out = {"ms_per_step": max_ms / steps,
           "value": whole_job_rate(tokens, max_ms, steps, world),
           "tokens_per_step": tokens, "wall_s": r["wall_s"],
           "gpu_launches": r["launches_per_step"] * steps}
    tensor = r["path"] == 1
    out["path"] = "tensor_core" if tensor else "cuda_core"
    names = ["prep", "state"]
    stage = max(range(2), key=lambda i: r["stage_ms"][i])
    stages = {}
    for i, nm in enumerate(names):
        # the state pass is tcgen05 for every input; the prep is tcgen05 for
        # bf16 inputs, and for fp32 inputs the split-operand Grams on
        # tcgen05 around an fp32 inverse on the CUDA cores
        tc = tensor and (nm == "state" or x["dtype"] == "bf16")
        key = "chunk_%s_%s" % (nm, "tc" if tc else "split")
        rf = roofline_of(x, nm, tensor, r["stage_ms"][i], peaks, peak_src)
        rf["kernel"] = key
        rf["traffic"] = traffic_record(key, w.name, os.path.join(
            ROOT, "momentum_delta_rule_gb300", "csrc", KERNEL_SOURCES[key]))
        stages[nm] = rf
    out["roofline"] = stages[names[stage]]
    out["roofline_call"] = roofline_of(x, "call", tensor, out["ms_per_step"], peaks, peak_src)
    out["roofline_call"]["what"] = "whole chunk forward (every kernel of the call)"
    out["stages"] = stages
    out["intermediate_bytes"] = {
        "bytes": intermediate_bytes(x),
        "what": "prepared blocks written by the prep kernel and read by the state pass "
                "(and, for fp32 inputs, the hi / lo bf16 parts of q, k, v); "
                "not algorithmic work"}
    out["config"] = config_of(w, x, "flushed before every timed step: 256 MiB written, "
                                    "then another 256 MiB read")
    out["dtype"] = "bf16" if x["dtype"] == "bf16" else "f32 (split bf16 operands)"
    if e2e and not args.no_e2e:
        n = max(3, min(steps, 10))
        e_ms, h2d, d2h = time_e2e(mdn, x, x_dev, n, 2)
        e_ms = max_over_ranks(e_ms, world, dev)
        out["e2e"] = {"value": whole_job_rate(tokens, e_ms, 1, world), "unit": "tokens/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": e_ms,
                      "streams": "copies in, kernels and copies out on three streams, "
                                 "two device buffer sets"}
    out["_x_dev"] = x_dev
    return out


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import momentum_delta_rule_gb300 as mdn
    mdn.lib()                                    # fails loudly if not built
    peaks, peak_src = load_peaks()
    if args.decode_only:
        d = time_decode(mdn, args.decode_steps, dev, peaks)
        if rank == 0:
            print(json.dumps(d), flush=True)
        return
    w = W.BY_NAME[args.workload]
    x = W.make_prefill(w)
    flush = L2Flush(L2_FLUSH_BYTES, dev)

    clocks = ClockSampler(local).start()
    m = measure_prefill(mdn, w, x, dev, args, args.steps, args.warmup, world, flush,
                        peaks, peak_src, e2e=False)
    clk = clocks.stop()
    x_dev = m.pop("_x_dev")
    tensor = m["path"] == "tensor_core"
    line = {"metric": "MDN chunkwise fwd tokens/s", "value": m["value"],
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": m["dtype"], "data": "synthetic", "config": m["config"],
            "gpu_launches": m["gpu_launches"], "path": m["path"],
            "roofline": m["roofline"], "roofline_call": m["roofline_call"],
            "stages": m["stages"], "intermediate_bytes": m["intermediate_bytes"],
            "clocks": clk, "peaks": peak_src}
    tokens = m["tokens_per_step"]
    if not args.no_vres and tensor:
        v_ms, v_bytes = time_vres(mdn, x_dev, max(3, min(args.steps, 10)), 2, flush)
        line["vres"] = {"what": "forward that also writes every token's residual "
                                "(mdn_chunk_fwd_vres)",
                        "ms_per_step": v_ms, "tokens_per_s": tokens / (v_ms / 1e3),
                        "extra_bytes_written": v_bytes,
                        "overhead_vs_forward": v_ms / m["ms_per_step"] - 1.0}
    if not args.no_inputs:
        line["inputs"] = time_inputs(mdn, x_dev, max(3, min(args.steps, 10)), 2, flush, peaks)
    if not args.no_backward:
        line["backward"] = time_backward(mdn, x, x_dev, max(3, min(args.steps, 10)), 2, flush,
                                         peaks)
        line["backward"]["ratio_to_forward"] = line["backward"]["ms_per_call"] / m["ms_per_step"]
    if not args.no_block and tensor:
        line["block"] = time_block(mdn, x_dev, max(3, min(args.steps, 10)), 2, flush)
    if not args.no_e2e:
        e_ms, h2d, d2h = time_e2e(mdn, x, x_dev, max(3, min(args.steps, 10)), 2)
        e_ms = max_over_ranks(e_ms, world, dev)
        line["e2e"] = {"value": whole_job_rate(tokens, e_ms, 1, world), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e_ms,
                       "streams": "copies in, kernels and copies out on three streams, "
                                  "two device buffer sets"}
    del x_dev
    if not args.no_decode:
        line["decode"] = time_decode(mdn, args.decode_steps, dev, peaks)
    if not args.no_other_workloads:
        others = {}
        n = max(3, min(args.steps, 5))
        for wo in W.ALL + [W.PREFILL_400M_FP32]:
            if wo.decode_steps or wo.name == w.name:
                continue
            xo = W.make_prefill(wo)
            mo = measure_prefill(mdn, wo, xo, dev, args, n, 3, world, flush, peaks, peak_src,
                                 e2e=wo.D == 128)
            mo.pop("_x_dev")
            mo["tokens_per_s"] = mo.pop("value")
            others[wo.name] = mo
        line["other_workloads"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_oracle(x, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
