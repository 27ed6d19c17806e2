"""Seeded synthetic inputs for the gated delta rule: the one module that both the
CUDA path's callers (tests, bench) and the float64 oracle draw their inputs from.

It holds no arithmetic of the method itself, only the input recipe. The draw order
and distributions follow the reproduction script on the mlx issue page
"mx.fast.gated_delta_update VJP: wrong gradient w.r.t. g (and ~1e-3 error on all
inputs) on the NAX path for Hk=16" (its `main()`): one `numpy.random.default_rng(seed)`
stream, drawn in the order

    q     = unit(N(0,1)) * Dk**-0.5              [B, T, Hk, Dk]
    k     = unit(N(0,1))                          [B, T, Hk, Dk]
    v     ~ N(0,1)                                [B, T, Hv, Dv]
    log g = -exp(N(mu, 0.5))                      [B, T, Hv]   mu = +2 strong, -2 weak
    beta  = sigmoid(N(0,1))                       [B, T, Hv]
    dy    ~ N(0,1)                                [B, T, Hv, Dv]
    S0    ~ N(0, 0.1)   (only when requested)     [B, Hv, Dv, Dk]
    dS_T  ~ N(0, 1)     (only when requested)     [B, Hv, Dv, Dk]

(normal(mean, std), as numpy takes it). The "half" decay mode gives value heads
h < Hv/2 the strong mean and the rest the weak one, the same for every batch row.

Gate inputs (make_gate_inputs). No page gives a recipe for the layer's raw gate inputs;
the reading taken draws, from its own stream, in the order

    a       ~ N(mu_a, 0.5)                       [B, T, Hv]   mu_a = +8 strong, -2 weak
    b       ~ N(0, 1)                            [B, T, Hv]   (the beta logits above)
    A_log   ~ N(0, 0.5)                          [Hv]
    dt_bias ~ N(0, 0.5)                          [Hv]
    dg      ~ N(0, 1), dbeta ~ N(0, 1)           [B, T, Hv]   (cotangents)

so that through the layer's gate map the mean log g lands near the strong (-8.4) and weak
(-0.15) profiles of the accuracy table. The "half" mode splits the heads as above.

Every array is returned as float32 holding exactly the value the kernels receive:
for bf16 workloads q, k, v, g, beta and dy are rounded to bf16 (round to nearest
even) and kept as float32 (an exact embedding). Widening to float64 for the oracle
is then exact, so the oracle sees bit-for-bit the inputs the GPU sees.
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    dtype: str = "f32"          # "f32" or "bf16": type of q, k, v, g, beta, dy and outputs
    decay: str = "weak"         # "weak", "strong" or "half"
    with_S0: bool = False
    with_dST: bool = False
    chunk: int = 64
    seed: int = 0

    def as_dict(self):
        return asdict(self)


# The workloads of the hot path, named by what they are.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 16, 2, 4, 32, 32, "f32", "weak"),
    "stress-strong": Workload("stress-strong", 1, 128, 16, 48, 128, 128, "f32", "strong"),
    "stress-weak": Workload("stress-weak", 1, 128, 16, 48, 128, 128, "f32", "weak"),
    "linattn-T256": Workload("linattn-T256", 1, 256, 16, 64, 192, 128, "bf16", "weak"),
    "linattn-T512": Workload("linattn-T512", 1, 512, 16, 64, 192, 128, "bf16", "weak"),
    "linattn-T1024": Workload("linattn-T1024", 1, 1024, 16, 64, 192, 128, "bf16", "weak"),
    "linattn-T2048": Workload("linattn-T2048", 1, 2048, 16, 64, 192, 128, "bf16", "weak"),
    "batched": Workload("batched", 8, 4096, 16, 32, 128, 128, "bf16", "half", True, True),
    "long": Workload("long", 1, 32768, 16, 64, 192, 128, "bf16", "weak", chunk=64),
    # the long-context layer's share of one GPU when its heads are split eight ways (2 of the 16
    # kv heads and their 8 value heads): few heads, so the sequence-parallel form has SMs to fill
    "long-tp8": Workload("long-tp8", 1, 32768, 2, 8, 192, 128, "bf16", "weak", chunk=64),
    # decode: one step of the same layer for B sequences, the state carried in and out (S0, S_T)
    "decode-B1": Workload("decode-B1", 1, 1, 16, 64, 192, 128, "bf16", "weak", True, False),
    "decode-B64": Workload("decode-B64", 64, 1, 16, 64, 192, 128, "bf16", "weak", True, False),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = ((u + bias) & np.uint32(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def _unit(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def make_inputs(w: Workload | None = None, **kw) -> dict:
    """Draw one workload's inputs. Either pass a Workload or its fields as keywords."""
    if w is None:
        w = Workload(name=kw.pop("name", "custom"), **kw)
    elif kw:
        w = Workload(**{**w.as_dict(), **kw})
    rng = np.random.default_rng(w.seed)
    B, T, Hk, Hv, Dk, Dv = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv

    q = (_unit(rng.standard_normal((B, T, Hk, Dk))) * Dk ** -0.5).astype(np.float32)
    k = _unit(rng.standard_normal((B, T, Hk, Dk))).astype(np.float32)
    v = rng.standard_normal((B, T, Hv, Dv)).astype(np.float32)
    if w.decay == "strong":
        mu = 2.0
    elif w.decay == "weak":
        mu = -2.0
    elif w.decay == "half":
        mu = np.where(np.arange(Hv) < Hv // 2, 2.0, -2.0)[None, None, :]
    else:
        raise ValueError(f"unknown decay mode {w.decay!r}")
    log_g = -np.exp(rng.normal(mu, 0.5, (B, T, Hv)))
    g = np.exp(log_g).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv))))).astype(np.float32)
    dy = rng.standard_normal((B, T, Hv, Dv)).astype(np.float32)
    S0 = rng.normal(0.0, 0.1, (B, Hv, Dv, Dk)).astype(np.float32) if w.with_S0 else None
    dS_T = rng.standard_normal((B, Hv, Dv, Dk)).astype(np.float32) if w.with_dST else None

    if w.dtype == "bf16":
        q, k, v, g, beta, dy = (round_to_bf16(a) for a in (q, k, v, g, beta, dy))
    elif w.dtype != "f32":
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return {"workload": w, "q": q, "k": k, "v": v, "g": g, "beta": beta, "dy": dy,
            "S0": S0, "dS_T": dS_T, "mean_log_g": float(log_g.mean())}


def make_gate_inputs(w: Workload) -> dict:
    """Draw the raw gate inputs of a workload (see the module docstring). a, b, dg, dbeta
    are rounded to bf16 for bf16 workloads; A_log and dt_bias are float32 parameters."""
    rng = np.random.default_rng(w.seed + 1)
    B, T, Hv = w.B, w.T, w.Hv
    if w.decay == "strong":
        mu = 8.0
    elif w.decay == "weak":
        mu = -2.0
    elif w.decay == "half":
        mu = np.where(np.arange(Hv) < Hv // 2, 8.0, -2.0)[None, None, :]
    else:
        raise ValueError(f"unknown decay mode {w.decay!r}")
    a = rng.normal(mu, 0.5, (B, T, Hv)).astype(np.float32)
    b = rng.standard_normal((B, T, Hv)).astype(np.float32)
    A_log = rng.normal(0.0, 0.5, Hv).astype(np.float32)
    dt_bias = rng.normal(0.0, 0.5, Hv).astype(np.float32)
    dg = rng.standard_normal((B, T, Hv)).astype(np.float32)
    dbeta = rng.standard_normal((B, T, Hv)).astype(np.float32)
    if w.dtype == "bf16":
        a, b, dg, dbeta = (round_to_bf16(x) for x in (a, b, dg, dbeta))
    elif w.dtype != "f32":
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return {"workload": w, "a": a, "b": b, "A_log": A_log, "dt_bias": dt_bias, "dg": dg, "dbeta": dbeta}
