"""Helpers for the GPU parity tests: run the CUDA library (through its binding) and the
float64 oracle on the same seeded inputs and compare every output by relative L2."""
from __future__ import annotations

import numpy as np

import oracle

# Tolerances (relative L2 over each whole output tensor), as stated for the hot path:
# float32 inputs <= 1e-5 on every output including dg under strong decay; bf16 inputs
# <= 5e-3 against the oracle run on the bf16-rounded values.
TOL = {"f32": 1e-5, "bf16": 5e-3}
OUTPUTS = ("y", "S_T", "ckpt", "dq", "dk", "dv", "dg", "dbeta", "dS0")


def to_device(inp, dev):
    import torch
    w = inp["workload"]
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    t = {}
    for n in ("q", "k", "v", "g", "beta", "dy"):
        t[n] = torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev).to(dt)
    for n in ("S0", "dS_T"):
        t[n] = None if inp[n] is None else torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev)
    return t


def run_gpu(inp, dev="cuda:0"):
    import torch
    import gated_delta_rule_22_gb300 as gdn
    w = inp["workload"]
    t = to_device(inp, dev)
    y, S_T, ckpt = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], chunk=w.chunk)
    gr = gdn.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ckpt, t["dy"], t["dS_T"], chunk=w.chunk)
    torch.cuda.synchronize()
    return {"y": y, "S_T": S_T, "ckpt": ckpt, **gr}


def to_numpy(out, names=OUTPUTS):
    return {n: out[n].double().cpu().numpy() for n in names if out.get(n) is not None}


def run_oracle(inp, nthreads=0):
    w = inp["workload"]
    f = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk,
                   nthreads=nthreads)
    b = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["dy"], inp["S0"],
                   inp["dS_T"], chunk=w.chunk, nthreads=nthreads)
    return {**f, **b}


def errors(got: dict, ref: dict) -> dict:
    return {n: oracle.rel_l2(got[n], ref[n]) for n in ref if n in got}


def log_errors(label: str, errs: dict) -> None:
    """Append one JSON line {label, errors} to the file named by $GDN_PARITY_LOG, if set (a
    record of the per-output errors of a parity run)."""
    import json
    import os
    path = os.environ.get("GDN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": label, "rel_l2": errs}) + "\n")


def group_outputs(out: dict, w, b: int, hk: int) -> dict:
    """The outputs of one (batch row, kv head) group, as numpy float64, laid out like a
    B=1, Hk=1 problem (matches oracle.group_slice)."""
    rep = w.Hv // w.Hk
    hs = slice(hk * rep, (hk + 1) * rep)
    sel = {
        "y": out["y"][b:b + 1, :, hs], "S_T": out["S_T"][b:b + 1, hs], "ckpt": out["ckpt"][b:b + 1, hs],
        "dq": out["dq"][b:b + 1, :, hk:hk + 1], "dk": out["dk"][b:b + 1, :, hk:hk + 1],
        "dv": out["dv"][b:b + 1, :, hs], "dg": out["dg"][b:b + 1, :, hs], "dbeta": out["dbeta"][b:b + 1, :, hs],
        "dS0": out["dS0"][b:b + 1, hs],
    }
    return {n: t.double().cpu().numpy() for n, t in sel.items()}


def oracle_group(inp, b: int, hk: int, nthreads=0) -> dict:
    w = inp["workload"]
    s = oracle.group_slice(inp, b, hk)
    f = oracle.fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], s["S0"], chunk=w.chunk, nthreads=nthreads)
    g = oracle.bwd(s["q"], s["k"], s["v"], s["g"], s["beta"], s["dy"], s["S0"], s["dS_T"], chunk=w.chunk,
                   nthreads=nthreads)
    return {**f, **g}
