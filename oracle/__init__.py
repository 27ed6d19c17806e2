"""float64 CPU oracle for the gated delta rule (forward + reverse-time VJP).

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU-baseline
leg may import this package; the product path (the CUDA library and its binding)
never does. The arithmetic lives in `gdn_oracle.c` (plain C, float64); this module
only compiles it with gcc and marshals numpy arrays through ctypes.

Functions
---------
fwd(q, k, v, g, beta, S0=None, chunk=64)  -> dict(y, S_T, ckpt)
bwd(q, k, v, g, beta, dy, S0=None, dS_T=None, chunk=64)
                                          -> dict(dq, dk, dv, dg, dbeta, dS0)
gates_fwd(a, b, A_log, dt_bias)           -> dict(g, beta)
gates_bwd(a, b, A_log, dt_bias, dg, dbeta) -> dict(da, db, dA_log, ddt_bias)
Layouts: q, k [B,T,Hk,Dk]; v, dy [B,T,Hv,Dv]; g, beta, a, b [B,T,Hv]; A_log, dt_bias [Hv];
states [B,Hv,Dv,Dk]; ckpt [B,Hv,NC,Dv,Dk] with ckpt[:, :, c] the state before step c*chunk.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

GCC_FLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp"]


class OracleShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int),
                ("Hv", ctypes.c_int), ("Dk", ctypes.c_int), ("Dv", ctypes.c_int),
                ("C", ctypes.c_int)]


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    cmd = ["gcc", *GCC_FLAGS, *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build(path: str, src: str) -> bool:
    return not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(src)


_P = ctypes.POINTER(ctypes.c_double)


def load(path: str | None = None):
    """Load (building if stale) the oracle library and declare its signatures."""
    if path is None:
        path = _LIB_PATH
        if _needs_build(path, _SRC):
            build()
    lib = ctypes.CDLL(path)
    lib.oracle_fwd.restype = ctypes.c_int
    lib.oracle_fwd.argtypes = [ctypes.POINTER(OracleShape)] + [_P] * 9 + [ctypes.c_int]
    lib.oracle_bwd.restype = ctypes.c_int
    lib.oracle_bwd.argtypes = [ctypes.POINTER(OracleShape)] + [_P] * 14 + [ctypes.c_int]
    lib.oracle_n_chunks.restype = ctypes.c_int
    lib.oracle_n_chunks.argtypes = [ctypes.POINTER(OracleShape)]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_gates_fwd.restype = ctypes.c_int
    lib.oracle_gates_fwd.argtypes = [ctypes.c_int, ctypes.c_int] + [_P] * 6
    lib.oracle_gates_bwd.restype = ctypes.c_int
    lib.oracle_gates_bwd.argtypes = [ctypes.c_int, ctypes.c_int] + [_P] * 10
    return lib


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _shape(q, v, chunk):
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    return OracleShape(B, T, Hk, Hv, Dk, Dv, chunk)


def max_threads(lib=None) -> int:
    return (lib or _lib()).oracle_max_threads()


def fwd(q, k, v, g, beta, S0=None, chunk=64, nthreads=0, lib=None):
    lib = lib or _lib()
    q, k, v, g, beta, S0 = (_f64(a) for a in (q, k, v, g, beta, S0))
    s = _shape(q, v, chunk)
    NC = (s.T + chunk - 1) // chunk
    y = np.empty(v.shape)
    S_T = np.empty((s.B, s.Hv, s.Dv, s.Dk))
    ckpt = np.empty((s.B, s.Hv, NC, s.Dv, s.Dk))
    rc = lib.oracle_fwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        _ptr(S0), _ptr(y), _ptr(S_T), _ptr(ckpt), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed with code {rc}")
    return {"y": y, "S_T": S_T, "ckpt": ckpt}


def bwd(q, k, v, g, beta, dy, S0=None, dS_T=None, chunk=64, nthreads=0, lib=None):
    lib = lib or _lib()
    q, k, v, g, beta, dy, S0, dS_T = (_f64(a) for a in (q, k, v, g, beta, dy, S0, dS_T))
    s = _shape(q, v, chunk)
    dq = np.empty(q.shape)
    dk = np.empty(k.shape)
    dv = np.empty(v.shape)
    dg = np.empty(g.shape)
    dbeta = np.empty(beta.shape)
    dS0 = np.empty((s.B, s.Hv, s.Dv, s.Dk))
    rc = lib.oracle_bwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        _ptr(S0), _ptr(dy), _ptr(dS_T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                        _ptr(dbeta), _ptr(dS0), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed with code {rc}")
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "dS0": dS0}


def gates_fwd(a, b, A_log, dt_bias, lib=None):
    lib = lib or _lib()
    a, b, A_log, dt_bias = (_f64(x) for x in (a, b, A_log, dt_bias))
    Hv = a.shape[-1]
    BT = a.size // Hv
    g = np.empty(a.shape)
    beta = np.empty(a.shape)
    rc = lib.oracle_gates_fwd(BT, Hv, _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g), _ptr(beta))
    if rc != 0:
        raise RuntimeError(f"oracle_gates_fwd failed with code {rc}")
    return {"g": g, "beta": beta}


def gates_bwd(a, b, A_log, dt_bias, dg, dbeta, lib=None):
    lib = lib or _lib()
    a, b, A_log, dt_bias, dg, dbeta = (_f64(x) for x in (a, b, A_log, dt_bias, dg, dbeta))
    Hv = a.shape[-1]
    BT = a.size // Hv
    da = np.empty(a.shape)
    db = np.empty(a.shape)
    dA_log = np.empty(Hv)
    ddt_bias = np.empty(Hv)
    rc = lib.oracle_gates_bwd(BT, Hv, _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(dg), _ptr(dbeta),
                              _ptr(da), _ptr(db), _ptr(dA_log), _ptr(ddt_bias))
    if rc != 0:
        raise RuntimeError(f"oracle_gates_bwd failed with code {rc}")
    return {"da": da, "db": db, "dA_log": dA_log, "ddt_bias": ddt_bias}


def loss(out_fwd, dy, dS_T=None) -> float:
    """The scalar whose gradient bwd returns: <dy, y> + <dS_T, S_T>."""
    L = float(np.sum(out_fwd["y"] * dy))
    if dS_T is not None:
        L += float(np.sum(out_fwd["S_T"] * dS_T))
    return L


def rel_l2(a, b) -> float:
    """Relative L2 error ||a - b|| / max(||b||, 1e-300) over the flattened arrays in
    float64 (the metric of the mlx issue #4614 repro script, `rel()`)."""
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def group_slice(inp: dict, b: int, hk: int) -> dict:
    """Inputs of one independent (batch row, kv head) group as a B=1, Hk=1 problem."""
    w = inp["workload"]
    rep = w.Hv // w.Hk
    hs = slice(hk * rep, (hk + 1) * rep)
    out = {
        "q": inp["q"][b:b + 1, :, hk:hk + 1], "k": inp["k"][b:b + 1, :, hk:hk + 1],
        "v": inp["v"][b:b + 1, :, hs], "g": inp["g"][b:b + 1, :, hs],
        "beta": inp["beta"][b:b + 1, :, hs], "dy": inp["dy"][b:b + 1, :, hs],
        "S0": None if inp["S0"] is None else inp["S0"][b:b + 1, hs],
        "dS_T": None if inp["dS_T"] is None else inp["dS_T"][b:b + 1, hs],
    }
    return out
