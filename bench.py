"""Benchmark of the gated delta rule training hot path (forward with checkpoints +
reverse-time VJP) on GB300, printing one JSON line.

A step is one gdn_fwd + one gdn_bwd over one batch of the workload (every step of the
hot path). Default workload: the 9B-like linear-attention layer of mlx-lm PR #1217's
performance table (B=1, Hk=16, Hv=64, Dk=192, Dv=128, T=2048, bf16 inputs, fp32 state,
weak decay, checkpoint interval 64), synthetic inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (the only reference this method has) on
the host cores, on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs its own copy of the workload (weak scaling; the
path shards over independent (batch row, kv head) groups with no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_synthetic as gs  # noqa: E402

METRIC = "gated-delta fwd+bwd tokens/s (Hv64,Dk192,Dv128,T2048 bf16); % of roofline"
UNIT = "tokens/s"
# FP32 FMA peak derived from unit counts and clock (152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz
# max SM clock): only a fallback when the live measurement (gdn_diag_fma_tflops) is not taken.
FP32_PEAK_DERIVED_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# Apple-silicon Metal VJP, fwd+bwd at this exact shape (149.8 ms for T=2048, mlx-lm
# PR #1217 performance table): another machine's number, quoted as context.
PAGES_TOKENS_PER_S = 2048 / 0.1498
# dram__bytes_read.sum + dram__bytes_write.sum per launch of a kernel, from one ncu capture,
# keyed by (hash of the kernel family's source files, KERNEL_FILES, when it was taken; kernel
# family); absent: not measured for the current sources. One capture per family, one launch
# after three warm-up steps of the bench workload (two DRAM metrics: a single-pass capture), e.g.
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none \
#       -k regex:^chunk_sweep -s 3 -c 1 python bench.py --steps 1 --warmup 3 --no-cpu-baseline
TRAFFIC = {
    ("6bca51b51f2b99a8", "chunk_prep"): 35600896 + 91542272,
    ("6bca51b51f2b99a8", "chunk_sweep"): 160030720 + 349309696,
    ("d71abe6af8b106d7", "chunk_dsweep"): 160391168 + 191910400,
    ("d71abe6af8b106d7", "chunk_grad"): 332331264 + 17533184,
    # the decode-B64 workload (`-k regex:^decode`, `--workload decode-B64`)
    ("5f1ef1aadd121d75", "decode"): 404523264 + 349300224,
}


def load_peaks():
    """HBM GB/s and dense bf16 TFLOP/s (sustained: the kernels run inside a long step)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "MEASURED_PEAKS.json (hbm_gbs, bf16_tflops_sustained): of measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1700.0, "source": "fallback 6.8 TB/s, 1.7 PFLOP/s sustained: of fallback"}


# The source files a kernel family's code and launch depend on (its translation unit, the
# shared headers, and the host code that builds its tensor maps): its traffic entry stays valid
# while these are unchanged.
KERNEL_FILES = {
    "chunk_prep": ("gdn_chunk.cu", "gdn_common.cuh", "gdn_umma.cuh", "gdn_api.cu"),
    "chunk_sweep": ("gdn_chunk.cu", "gdn_common.cuh", "gdn_umma.cuh", "gdn_api.cu"),
    "chunk_dsweep": ("gdn_chunk_bwd.cu", "gdn_common.cuh", "gdn_umma.cuh", "gdn_api.cu"),
    "chunk_grad": ("gdn_chunk_bwd.cu", "gdn_common.cuh", "gdn_umma.cuh", "gdn_api.cu"),
    "chunk_lite": ("gdn_chunk.cu", "gdn_common.cuh", "gdn_umma.cuh", "gdn_api.cu"),
    "decode": ("gdn_decode.cu", "gdn_common.cuh", "gdn_api.cu"),
    "segment_scan": ("gdn_segments.cu", "gdn_common.cuh", "gdn_api.cu"),
    "seq_fwd": ("gdn_fwd.cu", "gdn_common.cuh", "gdn_api.cu"),
    "seq_bwd": ("gdn_bwd.cu", "gdn_common.cuh", "gdn_api.cu"),
    "seq_reduce": ("gdn_bwd.cu", "gdn_common.cuh", "gdn_api.cu"),
}


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed: what the compiler sees."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return " ".join(text.split())


def kernel_source_hash(files=None):
    """Hash of the code (comments and layout aside) of the library's CUDA sources: all of
    them, or the named files."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_22_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")) and (files is None or f in files):
            h.update(f.encode())
            h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def traffic_of(name):
    """The DRAM traffic per launch measured for kernel family `name` on its current sources,
    or None."""
    files = KERNEL_FILES.get(name)
    return None if files is None else TRAFFIC.get((kernel_source_hash(files), name))


def flops_per_step(w, count=28):
    """Algorithmic FP32 flops: per token and value head, forward 7 Dv Dk (decay 1, S k 2,
    write 2, S q 2), backward 15 Dv Dk, plus one within-chunk re-computation of the state
    path (6 Dv Dk) that the checkpoint scheme prescribes: 28 in all (22 without it)."""
    return float(count) * w.B * w.T * w.Hv * w.Dv * w.Dk


def tensor_bytes(w):
    """HBM bytes of every tensor in the method's byte count of one fwd + bwd: inputs, outputs
    and the fp32 chunk-start checkpoints (S0 and dS_T only when the workload passes them)."""
    e = 2 if w.dtype == "bf16" else 4
    nc = -(-w.T // w.chunk)
    qk = w.B * w.T * w.Hk * w.Dk * e
    vv = w.B * w.T * w.Hv * w.Dv * e
    gate = w.B * w.T * w.Hv * e
    st = w.B * w.Hv * w.Dv * w.Dk * 4
    return {"q": qk, "k": qk, "v": vv, "g": gate, "beta": gate, "y": vv, "dy": vv, "dv": vv,
            "dq": qk, "dk": qk, "dg": gate, "dbeta": gate, "S0": st if w.with_S0 else 0, "S_T": st,
            "dS_T": st if w.with_dST else 0, "dS0": st, "ckpt": w.B * w.Hv * nc * w.Dv * w.Dk * 4}


# The tensors of each pass (forward: read q, k, v, g, beta, S0; write y, S_T and the
# checkpoints; backward: read q, k, v, g, beta, the checkpoints, dy, dS_T; write the six
# gradients), and the kernel each tensor is credited to: the one that reads it from (or writes
# it to) the caller's memory, or, where the design reads a tensor through an intermediate that
# another kernel derived from it, the kernel that consumes that intermediate. Every tensor of a
# pass is credited to exactly one kernel of that pass, so the kernels' algorithmic bytes add up
# to the pass's; intermediates (the chunkwise form's per-chunk operands, the backward's scratch)
# are credited to no kernel.
PASS_TENSORS = {
    "chunk_prep": ("q", "k", "v", "g", "beta"),
    "chunk_sweep": ("S0", "y", "S_T", "ckpt"),
    "chunk_dsweep": ("v", "beta", "dy", "dS_T", "dv", "dS0"),
    "chunk_grad": ("q", "k", "g", "ckpt", "dq", "dk", "dg", "dbeta"),
    "seq_fwd": ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt"),
    "seq_bwd": ("q", "k", "v", "g", "beta", "ckpt", "dy", "dS_T", "dv", "dS0"),
    "seq_reduce": ("dq", "dk", "dg", "dbeta"),
}


def bytes_per_step(w):
    """Algorithmic HBM bytes of one fwd + bwd: every input and output once per pass, plus the
    fp32 checkpoints written by the forward and read by the backward (scratch excluded)."""
    b = tensor_bytes(w)
    fwd = sum(b[n] for n in ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt"))
    bwd = sum(b[n] for n in ("q", "k", "v", "g", "beta", "ckpt", "dy", "dS_T", "dq", "dk", "dv", "dg", "dbeta",
                             "dS0"))
    return float(fwd + bwd)


def kernel_model(w):
    """Per kernel family: (algorithmic HBM bytes, tensor-core flops, FP32 flops) of one launch.
    Bytes: the tensors PASS_TENSORS credits to the kernel, once each. Tensor flops: the issued
    MMA products of the chunkwise form (2 per multiply-add). FP32 flops: the sequential
    kernels' (fp32 inputs), 7 Dv Dk per token and value head forward, 15 + 6 backward."""
    B, T, Hk, Hv, Dk, Dv, L = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, w.chunk
    NC = -(-T // L)
    ch, ck = B * Hv * NC, B * Hk * NC               # (chunk, value head), (chunk, kv head)
    rows = B * T * Hv
    tb = tensor_bytes(w)
    nb = {k: float(sum(tb[n] for n in v)) for k, v in PASS_TENSORS.items()}
    m = {}
    m["chunk_prep"] = (nb["chunk_prep"], ck * 2 * (2 * L * L * Dk) + ch * (2 * L * Dk * L), 0.0)
    # per chunk and value head: U = (T diag(beta)) V, W S^T, [Q; K] S^T, [P; KKm] Delta, the update
    m["chunk_sweep"] = (nb["chunk_sweep"], ch * (2 * L * L * Dv + 2 * L * Dv * Dk + 2 * 2 * L * Dv * Dk
                                                 + 2 * 2 * L * L * Dv + 2 * Dv * Dk * L), 0.0)
    m["chunk_dsweep"] = (nb["chunk_dsweep"], ch * (2 * 2 * L * Dv * Dk + 2 * L * Dv * L * 2 + 2 * Dv * Dk * L * 2), 0.0)
    m["chunk_grad"] = (
        nb["chunk_grad"],
        ck * 2 * (2 * L * L * Dk)     # [Q; K] K^T, once per (chunk, kv head)
        + ch * 2 * (2 * L * L * Dv + 2 * L * Dk * Dv + L * Dk * Dv + 2 * L * Dk * L
                    + 2 * L * Dk * L + L * L * L), 0.0)
    m["seq_fwd"] = (nb["seq_fwd"], 0.0, 7.0 * rows * Dv * Dk)
    m["seq_bwd"] = (nb["seq_bwd"], 0.0, 21.0 * rows * Dv * Dk)
    m["seq_reduce"] = (nb["seq_reduce"], 0.0, 0.0)
    return m


def kernel_roofline(name, ms, model, peaks):
    """The bound of one kernel launch taking `ms`: HBM bytes, tensor flops or FP32 flops,
    whichever needs the most time at its peak; achieved is that quantity over `ms`."""
    nbytes, tflops, fflops = model
    hbm, bf16 = peaks["hbm_gbs"], peaks["bf16_tflops"]
    fp32 = peaks.get("fp32_tflops", FP32_PEAK_DERIVED_TFLOPS)
    cands = [("hbm", nbytes / (hbm * 1e9), nbytes / (ms * 1e-3) / 1e9, hbm, "GB/s", nbytes),
             ("tensor", tflops / (bf16 * 1e12), tflops / (ms * 1e-3) / 1e12, bf16, "TFLOP/s", tflops),
             ("alu", fflops / (fp32 * 1e12), fflops / (ms * 1e-3) / 1e12, fp32, "TFLOP/s", fflops)]
    bound, t_min, achieved, peak, unit, amount = max(cands, key=lambda c: c[1])
    return {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "ms_per_launch": ms, "roofline_ms": t_min * 1e3, "per_launch": amount}


# ------------------------------------------------------------------ multi-rank helpers
def max_over_ranks(values, device, world):
    """Element-wise maximum of `values` (floats) over all ranks of the default process group
    (any backend: NCCL with a CUDA device, gloo with the CPU); the values themselves when
    world == 1. The slowest rank sets every timing of a weak-scaling run."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    m = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return [float(x) for x in m.tolist()]


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s of a weak-scaling run: every rank processes its own full workload
    (independent (batch row, kv head) groups, no data exchange) in the slowest rank's time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------- CPU baseline
def oracle_sample(w, seconds_budget, max_T=None):
    """Time the float64 oracle (forward + backward, all heads of the workload) on its first
    T' steps, T' grown until one run takes about `seconds_budget` seconds. Returns
    (tokens/s, threads, sample text, seconds of the timed run, T')."""
    import oracle
    lib = oracle.load()
    threads = oracle.max_threads(lib)
    max_T = max_T or w.T
    Tp = min(16, max_T)
    while True:
        inp = gs.make_inputs(w, T=Tp)
        t0 = time.perf_counter()
        oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk, lib=lib)
        oracle.bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["dy"], inp["S0"], inp["dS_T"],
                   chunk=w.chunk, lib=lib)
        dt = time.perf_counter() - t0
        if dt >= seconds_budget * 0.5 or Tp >= max_T:
            break
        Tp = min(max_T, max(Tp * 2, int(Tp * seconds_budget / max(dt, 1e-3) * 0.9)))
    sample = (f"oracle fwd+bwd over all {w.B * w.Hv} value heads, first {Tp} of {w.T} steps "
              f"(cost is linear in T), {threads} OpenMP threads")
    return w.B * Tp / dt, threads, sample, dt, Tp


# ---------------------------------------------------------------------------- runs
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    budget = max(1.0, 150.0 / (args.steps + args.warmup))
    _, threads, sample, _, Tp = oracle_sample(w, budget)
    import oracle
    lib = oracle.load()
    inp = gs.make_inputs(w, T=Tp)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk, lib=lib)
        oracle.bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["dy"], inp["S0"], inp["dS_T"],
                   chunk=w.chunk, lib=lib)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    value = w.B * Tp / per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, l2="host run"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, l2):
    return {"workload": f"{w.name}: B={w.B} T={w.T} Hk={w.Hk} Hv={w.Hv} Dk={w.Dk} Dv={w.Dv}, "
                        f"{w.dtype} inputs, fp32 state, {w.decay} decay, checkpoint interval {w.chunk}",
            "B": w.B, "T": w.T, "Hk": w.Hk, "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "chunk": w.chunk,
            "input_dtype": w.dtype, "decay": w.decay, "l2": l2}


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    import gated_delta_rule_22_gb300 as gdn

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gdn.load_library()

    inp = gs.make_inputs(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    names = ("q", "k", "v", "g", "beta", "dy")
    t = {n: torch.from_numpy(inp[n]).to(dev).to(dt) for n in names}
    for n in ("S0", "dS_T"):
        t[n] = None if inp[n] is None else torch.from_numpy(inp[n]).to(dev)
    B, T, Hk, Hv, Dk, Dv = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    S_T = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)
    grads = {"dq": torch.empty_like(t["q"]), "dk": torch.empty_like(t["k"]), "dv": torch.empty_like(t["v"]),
             "dg": torch.empty_like(t["g"]), "dbeta": torch.empty_like(t["beta"]),
             "dS0": torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)}
    shape = gdn.make_shape(B, T, Hk, Hv, Dk, Dv, w.chunk, 1 if w.dtype == "bf16" else 0)
    if args.segments == "auto":
        P = gdn.gdn_seg_choose(shape, torch.cuda.get_device_properties(dev).multi_processor_count)
        P = 0 if P <= 1 else P
    else:
        P = int(args.segments)
    RC = args.recompute and not P
    if RC:
        def new_saved(q, v):
            return gdn.new_rc_ckpt(q, v)
        ws = torch.empty(gdn.gdn_rc_bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    elif P:
        # the sequence-parallel form: its own saved buffer and workspace
        def new_saved(q, v):
            return torch.empty(gdn.gdn_seg_ckpt_bytes(shape, P), dtype=torch.uint8, device=dev)
        ws = torch.empty(gdn.gdn_seg_workspace_bytes(shape, P), dtype=torch.uint8, device=dev)
    else:
        def new_saved(q, v):
            return gdn.new_ckpt(q, v, w.chunk)
        ws = torch.empty(gdn.gdn_bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    ckpt = new_saved(t["q"], t["v"])
    stream = torch.cuda.current_stream()

    def fwd(d, y_, S_T_, ck):
        if RC:
            gdn.gdn_fwd_rc(d["q"], d["k"], d["v"], d["g"], d["beta"], t["S0"], y=y_, S_T=S_T_, ckpt=ck, workspace=ws)
        elif P:
            gdn.gdn_fwd_seg(d["q"], d["k"], d["v"], d["g"], d["beta"], t["S0"], P, y=y_, S_T=S_T_, ckpt=ck,
                            workspace=ws)
        else:
            gdn.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], t["S0"], w.chunk, y=y_, S_T=S_T_, ckpt=ck)

    def bwd(d, ck, out):
        if RC:
            gdn.gdn_bwd_rc(d["q"], d["k"], d["v"], d["g"], d["beta"], ck, d["dy"], t["dS_T"], workspace=ws, out=out)
        elif P:
            gdn.gdn_bwd_seg(d["q"], d["k"], d["v"], d["g"], d["beta"], ck, d["dy"], t["dS_T"], P, workspace=ws,
                            out=out)
        else:
            gdn.gdn_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], ck, d["dy"], t["dS_T"], w.chunk, workspace=ws,
                        out=out)

    def step():
        fwd(t, y, S_T, ckpt)
        bwd(t, ckpt, grads)

    step()
    torch.cuda.synchronize()
    peak_alloc = torch.cuda.max_memory_allocated(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 256 MiB > 129 MB L2

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(K):
            flush.fill_(i & 0xFF)                       # untimed: evicts L2 between steps
            ev[i][0].record(stream)
            fwd(t, y, S_T, ckpt)
            ev[i][1].record(stream)
            bwd(t, ckpt, grads)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    step_ms = fwd_ms + bwd_ms
    step_ms, fwd_ms, bwd_ms = max_over_ranks([step_ms, fwd_ms, bwd_ms], dev, world)
    clocks = clk.summary()

    # per-kernel device times: the same steps again with the library's event timing on
    gdn.gdn_timing_read()
    gdn.gdn_timing_enable(True)
    for i in range(K):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    ktimes = gdn.gdn_timing_read()
    gdn.gdn_timing_enable(False)
    launches_per_step = sum(n for n, _ in ktimes.values()) / K

    # end to end through the public API: pinned host inputs in, host results out
    host_in = {n: torch.from_numpy(inp[n]).to(dt).pin_memory() for n in names}
    out_shapes = [(n, x.shape, x.dtype) for n, x in list(grads.items()) + [("y", y), ("S_T", S_T)]]
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(int(np.prod(sh)) * torch.empty((), dtype=dty).element_size() for _, sh, dty in out_shapes)

    def run_e2e(K, pipelined):
        """K steps; each copies its inputs from pinned host memory to the device, runs gdn_fwd
        and gdn_bwd, and copies every result back to pinned host memory. Serial: one stream.
        Pipelined: uploads and downloads run on two more streams with two sets of device
        buffers, so that step i+1's upload and step i's download overlap each other and the
        neighbouring steps' kernels."""
        nslot = 2 if pipelined else 1
        comp = torch.cuda.current_stream()
        copy = torch.cuda.Stream() if pipelined else comp        # uploads
        down = torch.cuda.Stream() if pipelined else comp        # downloads (the other direction of the link)
        slots = []
        for _ in range(nslot):
            d_in = {n: torch.empty(host_in[n].shape, dtype=dt, device=dev) for n in names}
            d_out = {n: torch.empty(sh, dtype=dty, device=dev) for n, sh, dty in out_shapes}
            h_out = {n: torch.empty(sh, dtype=dty).pin_memory() for n, sh, dty in out_shapes}
            ck = new_saved(d_in["q"], d_in["v"])
            slots.append(dict(d_in=d_in, d_out=d_out, h_out=h_out, ck=ck, up=torch.cuda.Event(),
                              done=torch.cuda.Event(), down=torch.cuda.Event()))
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def upload(i):
            sl = slots[i % nslot]
            with torch.cuda.stream(copy):
                if i >= nslot:
                    copy.wait_event(sl["done"])          # step i - nslot no longer reads these inputs
                for n in names:
                    sl["d_in"][n].copy_(host_in[n], non_blocking=True)
                sl["up"].record(copy)

        start.record(copy)
        upload(0)
        for i in range(K):
            sl = slots[i % nslot]
            comp.wait_event(sl["up"])
            if i >= nslot:
                comp.wait_event(sl["down"])              # step i - nslot's results have left
            d, o = sl["d_in"], sl["d_out"]
            fwd(d, o["y"], o["S_T"], sl["ck"])
            bwd(d, sl["ck"], {n: o[n] for n in grads})
            sl["done"].record(comp)
            if i + 1 < K:
                upload(i + 1)
            with torch.cuda.stream(down):
                down.wait_event(sl["done"])
                for n in o:
                    sl["h_out"][n].copy_(o[n], non_blocking=True)
                sl["down"].record(down)
        copy.wait_stream(down)
        end.record(copy)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / K

    run_e2e(max(1, args.warmup), True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e2e_ms = run_e2e(K, True)
    e2e_serial_ms = run_e2e(K, False)
    e2e_ms, e2e_serial_ms = max_over_ranks([e2e_ms, e2e_serial_ms], dev, world)

    value = job_throughput(w.B * w.T, world, step_ms)
    peaks = load_peaks()
    fma = {"ffma": gdn.gdn_diag_fma_tflops(False), "ffma2": gdn.gdn_diag_fma_tflops(True)}
    peaks["fp32_tflops"] = max(fma.values())
    hbm_gbs = peaks["hbm_gbs"]
    f28, f22 = flops_per_step(w, 28), flops_per_step(w, 22)
    nbytes = bytes_per_step(w)
    src_hash = kernel_source_hash()
    model = kernel_model(w)
    kernels = {}
    for name, (n, ms) in ktimes.items():
        # per launch; the sequence-parallel form launches some families twice a step, and its
        # families are taken per step against the plain form's model of them
        per = K if (P or RC) else n
        kernels[name] = kernel_roofline(name, ms / per, model.get(name, (0.0, 0.0, 0.0)), peaks)
        kernels[name]["launches_per_step"] = n / K
        kernels[name]["share"] = ms / sum(t for _, t in ktimes.values())
        kernels[name]["traffic"] = traffic_of(name)
    dominant = max(kernels.values(), key=lambda k: k["share"])
    peak_src = {"hbm": peaks["source"], "tensor": peaks["source"],
                "alu": "measured live: gdn_diag_fma_tflops, best of scalar and packed FMA"}
    roof = {"bound": dominant["bound"], "achieved": dominant["achieved"], "peak": dominant["peak"],
            "unit": dominant["unit"], "frac": dominant["frac"], "traffic": traffic_of(dominant["kernel"]),
            "kernel": dominant["kernel"], "ms_per_launch": dominant["ms_per_launch"],
            "per_launch": dominant["per_launch"], "peak_source": peak_src[dominant["bound"]],
            "per_launch_note": "the method's tensors credited to this kernel (bench.PASS_TENSORS), once each; "
                               "intermediates not counted"}
    mma = sum(model[k][1] for k in kernels if k in model)
    # the whole step against the bound of the form that ran: the chunkwise form's (HBM bytes or
    # issued MMA flops at the sustained bf16 peak) when the tensor-core kernels ran, else the
    # sequential form's (HBM bytes or 28 Dv Dk FP32 flops per token and value head)
    t_hbm = nbytes / (hbm_gbs * 1e9)
    if mma > 0:
        t_cmp, form, cbound = mma / (peaks["bf16_tflops"] * 1e12), "chunkwise (tensor cores)", "tensor"
    else:
        t_cmp, form, cbound = f28 / (peaks["fp32_tflops"] * 1e12), "sequential (FP32 pipe)", "alu"
    t_step = max(t_hbm, t_cmp)
    roofline_step = {
        "form": form, "bound": "hbm" if t_hbm >= t_cmp else cbound, "bytes": nbytes,
        "mma_flops": mma, "fp32_flops_28": f28, "fp32_flops_22": f22, "roofline_ms": t_step * 1e3,
        "frac": t_step * 1e3 / step_ms, "achieved_gbs": nbytes / (step_ms * 1e-3) / 1e9, "hbm_peak_gbs": hbm_gbs,
        "note": "the step's time against max(algorithmic bytes / measured HBM bandwidth, the flops of the "
                "form that ran / that pipe's measured peak): the headline fraction",
    }
    context = None
    if mma > 0:
        t_seq = max(t_hbm, f28 / (peaks["fp32_tflops"] * 1e12))
        context = {"roofline_ms": t_seq * 1e3, "ratio_to_step": t_seq * 1e3 / step_ms,
                   "note": "context only: the sequential form's bound (28 Dv Dk FP32 flops per token and value "
                           "head at the measured FP32 rate); the chunkwise form that ran does other work, so "
                           "this is not a bound of this step"}
    NCk = -(-w.T // w.chunk)
    memory = {"ckpt_buffer_bytes": (gdn.gdn_rc_ckpt_bytes(shape) if RC else gdn.gdn_seg_ckpt_bytes(shape, P) if P
                                    else gdn.gdn_ckpt_bytes(shape)),
              "ckpt_states_bytes": w.B * w.Hv * NCk * w.Dv * w.Dk * 4,
              "bwd_workspace_bytes": (gdn.gdn_rc_bwd_workspace_bytes(shape) if RC else
                                      gdn.gdn_seg_workspace_bytes(shape, P) if P else gdn.gdn_bwd_workspace_bytes(shape)),
              "peak_allocated_bytes": peak_alloc,
              "note": "peak_allocated_bytes: torch's peak device allocation over one fwd + bwd step "
                      "(inputs, outputs, saved buffer and workspace)"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGES_TOKENS_PER_S if w.name == "linattn-T2048" else None,
        "vs_baseline_note": "ratio to the Apple-silicon Metal VJP figure on the pages (another machine; context)",
        "dtype": "bf16" if mma > 0 else "f32",
        "dtype_note": ("bf16 tensor-core operands, f32 state and accumulation" if mma > 0
                       else "f32 arithmetic on the sequential kernels"),
        "data": "synthetic",
        "config": {**config_of(w, l2="flushed between steps by an untimed 256 MiB write"),
                   **({"segments": P, "form": "sequence-parallel (gdn_fwd_seg / gdn_bwd_seg)",
                       "kernels_note": "per-family figures are per step, against the plain form's model"}
                      if P else {}),
                   **({"form": "re-computation (gdn_fwd_rc / gdn_bwd_rc: the saved buffer holds checkpoints "
                               "and residuals; the backward forms the per-chunk products again)",
                       "kernels_note": "per-family figures are per step, against the plain form's model"}
                      if RC else {})},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "roofline": roof,
        "roofline_step": roofline_step,
        "sequential_form_context": context,
        "fp32_peak_tflops_measured": fma,
        "kernels": kernels,
        "memory": memory,
        "e2e": {"value": job_throughput(w.B * w.T, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "mode": "each step uploads its inputs from pinned host memory and downloads all results; "
                        "uploads and downloads on two more streams with two buffer sets overlap the kernels "
                        "of the neighbouring steps and each other",
                "serial": {"value": job_throughput(w.B * w.T, world, e2e_serial_ms), "ms_per_step": e2e_serial_ms,
                           "mode": "one stream: upload, kernels, download in sequence"}},
        "gpu_launches": int(round(launches_per_step * K)),
        "clocks": clocks,
        "kernel_sources": src_hash,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, threads, sample, _, _ = oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


DECODE_METRIC = "gated-delta decode tokens/s (one step, state in and out; Hv64,Dk192,Dv128 bf16)"


def run_decode(args, w):
    """One decode step of B sequences per call: gdn_fwd with T = 1, no saved buffer, the state
    passed in (S0) and returned (S_T), ping-ponged between two device arrays. HBM-bound: each
    step reads and writes every state once (2 B Hv Dv Dk fp32) plus the step's small tensors."""
    import torch
    import gated_delta_rule_22_gb300 as gdn
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    gdn.load_library()
    inp = gs.make_inputs(w)
    dt = torch.bfloat16
    names = ("q", "k", "v", "g", "beta")
    t = {n: torch.from_numpy(inp[n]).to(dev).to(dt) for n in names}
    S = [torch.from_numpy(inp["S0"]).to(dev), torch.empty_like(torch.from_numpy(inp["S0"])).to(dev)]
    y = torch.empty((w.B, 1, w.Hv, w.Dv), dtype=dt, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], S[i & 1], w.chunk, y=y, S_T=S[(i + 1) & 1],
                    want_ckpt=False)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    K = max(args.steps, 50)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    with ClockSampler(dev.index) as clk:
        for i in range(K):
            flush.fill_(i & 0xFF)                       # untimed: evicts L2 between steps
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    gdn.gdn_timing_read()
    gdn.gdn_timing_enable(True)
    for i in range(K):
        flush.fill_(i & 0xFF)
        step(i)
    torch.cuda.synchronize()
    kt = gdn.gdn_timing_read()
    gdn.gdn_timing_enable(False)
    # end to end: the step's inputs up from pinned host memory, y back down; the state stays
    host_in = {n: torch.from_numpy(inp[n]).to(dt).pin_memory() for n in names}
    h_y = torch.empty(y.shape, dtype=dt).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = y.numel() * y.element_size()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        for n in names:
            t[n].copy_(host_in[n], non_blocking=True)
        step(i)
        h_y.copy_(y, non_blocking=True)
    end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = start.elapsed_time(end) / K
    e = 2
    state = w.B * w.Hv * w.Dv * w.Dk * 4
    nbytes = 2 * state + w.B * (2 * w.Hk * w.Dk + 2 * w.Hv * w.Dv + 2 * w.Hv) * e
    peaks = load_peaks()
    kname = "decode" if "decode" in kt else "seq_fwd"
    n_fwd, ms_fwd = kt.get(kname, (K, ms * K))
    per_launch = ms_fwd / n_fwd
    achieved = nbytes / (per_launch * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": w.B / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**config_of(w, l2="flushed between steps by an untimed 256 MiB write"), "form": "decode"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic_of(kname), "kernel": kname,
                     "ms_per_launch": per_launch, "per_launch": nbytes,
                     "per_launch_note": "the state read and written once (fp32), q, k, v, g, beta read and y written once",
                     "peak_source": peaks["source"]},
        "kernels": {k: {"launches_per_step": n / K, "ms_per_launch": m / n} for k, (n, m) in kt.items()},
        "e2e": {"value": w.B / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "mode": "one stream: the step's inputs up, the step, y down; the state stays on the device"},
        "gpu_launches": int(round(sum(n for n, _ in kt.values()))),
        "clocks": clk.summary(),
        "kernel_sources": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="linattn-T2048", choices=sorted(gs.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--segments", default="0",
                    help="time the sequence-parallel form with this many segments (0: the plain calls; "
                         "auto: the count gdn_seg_choose gives for this GPU)")
    ap.add_argument("--recompute", action="store_true",
                    help="time the re-computation mode (saved buffer: checkpoints and residuals only)")
    args = ap.parse_args()
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    w = gs.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif w.T == 1:
        run_decode(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
