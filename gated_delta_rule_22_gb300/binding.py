"""Thin ctypes binding of libgdn.so (include/gdn.h). Argument marshalling only.

Every computation happens in the CUDA kernels behind the C ABI; PyTorch is used here
only to hold device memory and to supply the current CUDA stream. If the compiled
library is missing, loading fails with an ImportError; there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "gdn.h")

GDN_F32, GDN_BF16 = 0, 1
GDN_OK = 0
GDN_ERR_UNSUPPORTED_SHAPE = -3


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
                ("Dk", ctypes.c_int), ("Dv", ctypes.c_int), ("chunk", ctypes.c_int), ("dtype", ctypes.c_int)]


class GdnKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("ms", ctypes.c_double)]


class GdnError(RuntimeError):
    def __init__(self, fn, code, lib):
        self.code = code
        msg = lib.gdn_strerror(code).decode()
        detail = lib.gdn_last_error().decode()
        super().__init__(f"{fn} returned {code}: {msg}" + (f" [{detail}]" if detail else ""))


_VP = ctypes.c_void_p
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgdn.so and declare the signatures of include/gdn.h."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    SP = ctypes.POINTER(GdnShape)
    lib.gdn_ckpt_bytes.restype = ctypes.c_size_t
    lib.gdn_ckpt_bytes.argtypes = [SP]
    lib.gdn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_bwd_workspace_bytes.argtypes = [SP]
    lib.gdn_fwd.restype = ctypes.c_int
    _SZ = ctypes.c_size_t
    lib.gdn_fwd.argtypes = [SP] + [_VP] * 9 + [_SZ, _VP]
    lib.gdn_bwd.restype = ctypes.c_int
    lib.gdn_bwd.argtypes = [SP] + [_VP] * 6 + [_SZ] + [_VP] * 9 + [_SZ, _VP]
    lib.gdn_bwd_noalloc.restype = ctypes.c_int
    lib.gdn_bwd_noalloc.argtypes = [SP] + [_VP] * 6 + [_SZ] + [_VP] * 9
    lib.gdn_seg_choose.restype = ctypes.c_int
    lib.gdn_seg_choose.argtypes = [SP, ctypes.c_int]
    lib.gdn_seg_ckpt_bytes.restype = ctypes.c_size_t
    lib.gdn_seg_ckpt_bytes.argtypes = [SP, ctypes.c_int]
    lib.gdn_seg_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_seg_workspace_bytes.argtypes = [SP, ctypes.c_int]
    lib.gdn_fwd_seg.restype = ctypes.c_int
    lib.gdn_fwd_seg.argtypes = [SP, ctypes.c_int] + [_VP] * 9 + [_SZ, _VP, _SZ, _VP]
    lib.gdn_bwd_seg.restype = ctypes.c_int
    lib.gdn_bwd_seg.argtypes = [SP, ctypes.c_int] + [_VP] * 6 + [_SZ] + [_VP] * 9 + [_SZ, _VP]
    lib.gdn_infer_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_infer_workspace_bytes.argtypes = [SP]
    lib.gdn_fwd_infer.restype = ctypes.c_int
    lib.gdn_fwd_infer.argtypes = [SP] + [_VP] * 9 + [_SZ, _VP]
    for name in ("gdn_rc_ckpt_bytes", "gdn_rc_fwd_workspace_bytes", "gdn_rc_bwd_workspace_bytes"):
        getattr(lib, name).restype = ctypes.c_size_t
        getattr(lib, name).argtypes = [SP]
    lib.gdn_fwd_rc.restype = ctypes.c_int
    lib.gdn_fwd_rc.argtypes = [SP] + [_VP] * 9 + [_SZ, _VP, _SZ, _VP]
    lib.gdn_bwd_rc.restype = ctypes.c_int
    lib.gdn_bwd_rc.argtypes = [SP] + [_VP] * 6 + [_SZ] + [_VP] * 9 + [_SZ, _VP]
    lib.gdn_gates_fwd.restype = ctypes.c_int
    lib.gdn_gates_fwd.argtypes = [SP] + [_VP] * 7
    lib.gdn_gates_bwd.restype = ctypes.c_int
    lib.gdn_gates_bwd.argtypes = [SP] + [_VP] * 11
    lib.gdn_strerror.restype = ctypes.c_char_p
    lib.gdn_strerror.argtypes = [ctypes.c_int]
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_device_status.restype = ctypes.c_int
    lib.gdn_device_status.argtypes = []
    lib.gdn_version.restype = ctypes.c_int
    lib.gdn_version.argtypes = []
    lib.gdn_timing_enable.restype = ctypes.c_int
    lib.gdn_timing_enable.argtypes = [ctypes.c_int]
    lib.gdn_timing_read.restype = ctypes.c_int
    lib.gdn_timing_read.argtypes = [ctypes.POINTER(GdnKernelTime), ctypes.c_int]
    lib.gdn_debug_wait_probe.restype = ctypes.c_int
    lib.gdn_debug_wait_probe.argtypes = [ctypes.c_uint, _VP]
    lib.gdn_diag_fma_tflops.restype = ctypes.c_int
    lib.gdn_diag_fma_tflops.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    if path == LIB_PATH:
        _lib = lib
    return lib


def header_functions(header: str = HEADER):
    """Names of the functions declared in include/gdn.h."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return GDN_F32
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; the library takes float32 or bfloat16")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(name, t, shape, dtype, device):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _require_cuda(t):
    """The library takes device pointers only: a host tensor here would reach the kernels as a
    host address. The other tensors of a call are checked to be on t's device."""
    if t.device.type != "cuda":
        raise ValueError(f"tensors are on {t.device}; the library takes CUDA tensors")


def make_shape(B, T, Hk, Hv, Dk, Dv, chunk=64, dtype=GDN_F32) -> GdnShape:
    return GdnShape(B, T, Hk, Hv, Dk, Dv, chunk, dtype)


def _stream(stream, device=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def gdn_timing_enable(on: bool = True) -> None:
    """Per-kernel device timing of the library's own launches (a diagnostic)."""
    load_library().gdn_timing_enable(1 if on else 0)


def gdn_timing_read() -> dict:
    """{kernel family: (launches, summed ms)} since the last read; clears the record."""
    lib = load_library()
    buf = (GdnKernelTime * 32)()
    n = lib.gdn_timing_read(buf, 32)
    if n < 0:
        raise GdnError("gdn_timing_read", n, lib)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms) for i in range(min(n, 32))}


def gdn_ckpt_bytes(shape: GdnShape) -> int:
    return load_library().gdn_ckpt_bytes(ctypes.byref(shape))


def gdn_bwd_workspace_bytes(shape: GdnShape) -> int:
    return load_library().gdn_bwd_workspace_bytes(ctypes.byref(shape))


def _room(t) -> int:
    """Bytes of t's storage from its first element on."""
    return t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()


def new_ckpt(q, v, chunk=64):
    """The saved-for-backward buffer of gdn_fwd for inputs shaped like q and v: one fp32
    allocation of gdn_ckpt_bytes bytes, returned as its leading [B, Hv, NC, Dv, Dk] view of
    chunk-start states (the per-step residuals v - u follow in the same storage)."""
    torch = _torch()
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    NC = -(-T // (chunk or 64))
    need = gdn_ckpt_bytes(_shape_of(q, v, chunk))
    buf = torch.empty(-(-need // 4), dtype=torch.float32, device=q.device)
    return buf[: B * Hv * NC * Dv * Dk].view(B, Hv, NC, Dv, Dk)


def _check_ckpt(ckpt, q, v, chunk):
    torch = _torch()
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    NC = -(-T // (chunk or 64))
    _check("ckpt", ckpt, (B, Hv, NC, Dv, Dk), torch.float32, q.device)
    need = gdn_ckpt_bytes(_shape_of(q, v, chunk))
    if _room(ckpt) < need:
        raise ValueError(f"ckpt: its storage holds {_room(ckpt)} bytes from the first state on, "
                         f"gdn_ckpt_bytes = {need} (allocate it with new_ckpt)")


def _shape_of(q, v, chunk):
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    return make_shape(B, T, Hk, Hv, Dk, Dv, chunk, _dtype_code(q))


def gdn_fwd(q, k, v, g, beta, S0=None, chunk=64, *, y=None, S_T=None, ckpt=None, want_S_T=True,
            want_ckpt=True, stream=None):
    """y, S_T, ckpt = gdn_fwd(q, k, v, g, beta[, S0]) on CUDA tensors (see include/gdn.h).
    ckpt is the [B, Hv, NC, Dv, Dk] view of the saved-for-backward buffer (new_ckpt), or None
    with want_ckpt=False (inference / decode: nothing is saved)."""
    torch = _torch()
    lib = load_library()
    shape = _shape_of(q, v, chunk)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv))):
        _check(name, t, shp, dt, dev)
    if S0 is not None:
        _check("S0", S0, (B, Hv, Dv, Dk), torch.float32, dev)
    if y is not None:
        _check("y", y, (B, T, Hv, Dv), dt, dev)
    if S_T is not None:
        _check("S_T", S_T, (B, Hv, Dv, Dk), torch.float32, dev)
    if ckpt is not None:
        _check_ckpt(ckpt, q, v, chunk)
    _require_cuda(q)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if S_T is None and want_S_T:
        S_T = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)
    if ckpt is None and want_ckpt:
        ckpt = new_ckpt(q, v, chunk)
    rc = lib.gdn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                     _ptr(y), _ptr(S_T), _ptr(ckpt), 0 if ckpt is None else _room(ckpt), _stream(stream, dev))
    if rc != GDN_OK:
        raise GdnError("gdn_fwd", rc, lib)
    return y, S_T, ckpt


def _bwd_prepare(q, k, v, g, beta, ckpt, dy, dS_T, chunk, out, want_dS0, workspace=None):
    """Checks of a backward call's tensors (all before anything is allocated or launched), then
    the output dict (the caller's, or new tensors). Returns (shape, out)."""
    torch = _torch()
    shape = _shape_of(q, v, chunk)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv)), ("dy", dy, (B, T, Hv, Dv))):
        _check(name, t, shp, dt, dev)
    _check_ckpt(ckpt, q, v, chunk)
    if dS_T is not None:
        _check("dS_T", dS_T, (B, Hv, Dv, Dk), torch.float32, dev)
    if out is not None:
        for name, shp in (("dq", q.shape), ("dk", q.shape), ("dv", (B, T, Hv, Dv)), ("dg", (B, T, Hv)),
                          ("dbeta", (B, T, Hv))):
            if out.get(name) is None:
                raise ValueError(f"out lacks {name}")
            _check(name, out[name], shp, dt, dev)
        if out.get("dS0") is not None:
            _check("dS0", out["dS0"], (B, Hv, Dv, Dk), torch.float32, dev)
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError(f"workspace must be a contiguous tensor on {dev}")
    _require_cuda(q)
    if out is None:
        out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
               "dg": torch.empty_like(g), "dbeta": torch.empty_like(beta),
               "dS0": torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev) if want_dS0 else None}
    return shape, out


def gdn_bwd(q, k, v, g, beta, ckpt, dy, dS_T=None, chunk=64, *, workspace=None, out=None,
            want_dS0=True, stream=None):
    """dict(dq, dk, dv, dg, dbeta, dS0) = gdn_bwd(...) on CUDA tensors (see include/gdn.h).
    workspace: a device tensor of at least gdn_bwd_workspace_bytes bytes, or None (allocated
    here for this call)."""
    torch = _torch()
    lib = load_library()
    shape, out = _bwd_prepare(q, k, v, g, beta, ckpt, dy, dS_T, chunk, out, want_dS0, workspace)
    if workspace is None:
        need = lib.gdn_bwd_workspace_bytes(ctypes.byref(shape))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.gdn_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ckpt),
                     _room(ckpt), _ptr(dy), _ptr(dS_T), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                     _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out.get("dS0")), _ptr(workspace),
                     workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    if rc != GDN_OK:
        raise GdnError("gdn_bwd", rc, lib)
    return out


def gdn_seg_choose(shape: GdnShape, sm_count: int) -> int:
    return int(load_library().gdn_seg_choose(ctypes.byref(shape), sm_count))


def gdn_seg_ckpt_bytes(shape: GdnShape, segments: int) -> int:
    return int(load_library().gdn_seg_ckpt_bytes(ctypes.byref(shape), segments))


def gdn_seg_workspace_bytes(shape: GdnShape, segments: int) -> int:
    return int(load_library().gdn_seg_workspace_bytes(ctypes.byref(shape), segments))


def gdn_infer_workspace_bytes(shape: GdnShape) -> int:
    return int(load_library().gdn_infer_workspace_bytes(ctypes.byref(shape)))


def gdn_fwd_infer(q, k, v, g, beta, S0=None, *, y=None, S_T=None, workspace=None, want_S_T=True, stream=None):
    """y, S_T = gdn_fwd_infer(q, k, v, g, beta[, S0]): the inference forward on the tensor cores
    (include/gdn.h): nothing saved; the per-chunk products go to `workspace`
    (gdn_infer_workspace_bytes, allocated here when None)."""
    torch = _torch()
    lib = load_library()
    shape = _shape_of(q, v, 64)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv))):
        _check(name, t, shp, dt, dev)
    if S0 is not None:
        _check("S0", S0, (B, Hv, Dv, Dk), torch.float32, dev)
    _require_cuda(q)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if S_T is None and want_S_T:
        S_T = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)
    workspace = _workspace(workspace, lib.gdn_infer_workspace_bytes(ctypes.byref(shape)), dev)
    rc = lib.gdn_fwd_infer(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(y),
                           _ptr(S_T), _ptr(workspace), _room(workspace), _stream(stream, dev))
    if rc != GDN_OK:
        raise GdnError("gdn_fwd_infer", rc, lib)
    return y, S_T


def gdn_rc_ckpt_bytes(shape: GdnShape) -> int:
    return int(load_library().gdn_rc_ckpt_bytes(ctypes.byref(shape)))


def gdn_rc_fwd_workspace_bytes(shape: GdnShape) -> int:
    return int(load_library().gdn_rc_fwd_workspace_bytes(ctypes.byref(shape)))


def gdn_rc_bwd_workspace_bytes(shape: GdnShape) -> int:
    return int(load_library().gdn_rc_bwd_workspace_bytes(ctypes.byref(shape)))


def new_rc_ckpt(q, v):
    """The saved buffer of gdn_fwd_rc for inputs shaped like q and v (gdn_rc_ckpt_bytes bytes),
    returned as its leading [B, Hv, NC, Dv, Dk] fp32 view of chunk-start states."""
    torch = _torch()
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    NC = -(-T // 64)
    need = gdn_rc_ckpt_bytes(_shape_of(q, v, 64))
    if need == 0:
        raise GdnError("gdn_rc_ckpt_bytes", GDN_ERR_UNSUPPORTED_SHAPE, load_library())
    buf = torch.empty(-(-need // 4), dtype=torch.float32, device=q.device)
    return buf[: B * Hv * NC * Dv * Dk].view(B, Hv, NC, Dv, Dk)


def _workspace(t, need, dev):
    torch = _torch()
    if t is None:
        return torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if t.device != dev or not t.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {dev}")
    return t


def gdn_fwd_rc(q, k, v, g, beta, S0=None, *, y=None, S_T=None, ckpt=None, workspace=None, want_S_T=True,
               stream=None):
    """y, S_T, ckpt = gdn_fwd_rc(...): the forward of the re-computation mode (include/gdn.h):
    ckpt holds only the chunk-start states and the residuals (new_rc_ckpt when None); the
    per-chunk products go to `workspace` (gdn_rc_fwd_workspace_bytes, allocated here when None)."""
    torch = _torch()
    lib = load_library()
    shape = _shape_of(q, v, 64)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv))):
        _check(name, t, shp, dt, dev)
    if S0 is not None:
        _check("S0", S0, (B, Hv, Dv, Dk), torch.float32, dev)
    _require_cuda(q)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if S_T is None and want_S_T:
        S_T = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)
    if ckpt is None:
        ckpt = new_rc_ckpt(q, v)
    workspace = _workspace(workspace, lib.gdn_rc_fwd_workspace_bytes(ctypes.byref(shape)), dev)
    rc = lib.gdn_fwd_rc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(y),
                        _ptr(S_T), _ptr(ckpt), _room(ckpt), _ptr(workspace), _room(workspace), _stream(stream, dev))
    if rc != GDN_OK:
        raise GdnError("gdn_fwd_rc", rc, lib)
    return y, S_T, ckpt


def gdn_bwd_rc(q, k, v, g, beta, ckpt, dy, dS_T=None, *, workspace=None, out=None, want_dS0=True, stream=None):
    """dict(dq, dk, dv, dg, dbeta, dS0) = gdn_bwd_rc(...): the backward of the re-computation
    mode for the saved buffer of gdn_fwd_rc (include/gdn.h)."""
    torch = _torch()
    lib = load_library()
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    shape = _shape_of(q, v, 64)
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv)), ("dy", dy, (B, T, Hv, Dv))):
        _check(name, t, shp, dt, dev)
    if dS_T is not None:
        _check("dS_T", dS_T, (B, Hv, Dv, Dk), torch.float32, dev)
    _require_cuda(q)
    if out is None:
        out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
               "dg": torch.empty_like(g), "dbeta": torch.empty_like(beta),
               "dS0": torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev) if want_dS0 else None}
    workspace = _workspace(workspace, lib.gdn_rc_bwd_workspace_bytes(ctypes.byref(shape)), dev)
    rc = lib.gdn_bwd_rc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ckpt),
                        _room(ckpt), _ptr(dy), _ptr(dS_T), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                        _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out.get("dS0")), _ptr(workspace),
                        _room(workspace), _stream(stream, dev))
    if rc != GDN_OK:
        raise GdnError("gdn_bwd_rc", rc, lib)
    return out


def gdn_fwd_seg(q, k, v, g, beta, S0=None, segments=2, *, y=None, S_T=None, ckpt=None, workspace=None,
                want_S_T=True, stream=None):
    """y, S_T, ckpt = gdn_fwd_seg(q, k, v, g, beta[, S0], segments) on CUDA tensors: the
    sequence-parallel forward (see include/gdn.h). ckpt is a uint8 device tensor of
    gdn_seg_ckpt_bytes bytes (allocated here when None); workspace likewise
    (gdn_seg_workspace_bytes, allocated here for this call when None)."""
    torch = _torch()
    lib = load_library()
    shape = _shape_of(q, v, 64)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv))):
        _check(name, t, shp, dt, dev)
    if S0 is not None:
        _check("S0", S0, (B, Hv, Dv, Dk), torch.float32, dev)
    if y is not None:
        _check("y", y, (B, T, Hv, Dv), dt, dev)
    if S_T is not None:
        _check("S_T", S_T, (B, Hv, Dv, Dk), torch.float32, dev)
    for name, t in (("ckpt", ckpt), ("workspace", workspace)):
        if t is not None and (t.device != dev or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous tensor on {dev}")
    _require_cuda(q)
    need_ck = lib.gdn_seg_ckpt_bytes(ctypes.byref(shape), segments)
    need_ws = lib.gdn_seg_workspace_bytes(ctypes.byref(shape), segments)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=dt, device=dev)
    if S_T is None and want_S_T:
        S_T = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)
    if ckpt is None:
        ckpt = torch.empty(max(need_ck, 16), dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = torch.empty(max(need_ws, 16), dtype=torch.uint8, device=dev)
    rc = lib.gdn_fwd_seg(ctypes.byref(shape), segments, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                         _ptr(y), _ptr(S_T), _ptr(ckpt), _room(ckpt), _ptr(workspace), _room(workspace),
                         _stream(stream, dev))
    if rc != GDN_OK:
        raise GdnError("gdn_fwd_seg", rc, lib)
    return y, S_T, ckpt


def gdn_bwd_seg(q, k, v, g, beta, ckpt, dy, dS_T=None, segments=2, *, workspace=None, out=None, want_dS0=True,
                stream=None):
    """dict(dq, dk, dv, dg, dbeta, dS0) = gdn_bwd_seg(...): the sequence-parallel backward for
    the saved buffer of gdn_fwd_seg with the same segments (see include/gdn.h)."""
    torch = _torch()
    lib = load_library()
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    dev, dt = q.device, q.dtype
    shape = _shape_of(q, v, 64)
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("v", v, (B, T, Hv, Dv)),
                         ("g", g, (B, T, Hv)), ("beta", beta, (B, T, Hv)), ("dy", dy, (B, T, Hv, Dv))):
        _check(name, t, shp, dt, dev)
    if dS_T is not None:
        _check("dS_T", dS_T, (B, Hv, Dv, Dk), torch.float32, dev)
    for name, t in (("ckpt", ckpt), ("workspace", workspace)):
        if t is not None and (t.device != dev or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous tensor on {dev}")
    _require_cuda(q)
    if out is None:
        out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
               "dg": torch.empty_like(g), "dbeta": torch.empty_like(beta),
               "dS0": torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev) if want_dS0 else None}
    if workspace is None:
        need = lib.gdn_seg_workspace_bytes(ctypes.byref(shape), segments)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib.gdn_bwd_seg(ctypes.byref(shape), segments, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ckpt),
                         _room(ckpt), _ptr(dy), _ptr(dS_T), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                         _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out.get("dS0")), _ptr(workspace),
                         _room(workspace), _stream(stream, dev))
    if rc != GDN_OK:
        raise GdnError("gdn_bwd_seg", rc, lib)
    return out


def gdn_bwd_noalloc(q, k, v, g, beta, ckpt, dy, dS_T=None, chunk=64, *, out=None, want_dS0=True,
                    stream=None):
    """gdn_bwd with the library's fixed device scratch instead of a workspace (see
    include/gdn.h: calls that overlap on one GPU race on that scratch). Pass `out` to
    allocate nothing here either."""
    lib = load_library()
    shape, out = _bwd_prepare(q, k, v, g, beta, ckpt, dy, dS_T, chunk, out, want_dS0)
    rc = lib.gdn_bwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ckpt),
                             _room(ckpt), _ptr(dy), _ptr(dS_T), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                             _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out.get("dS0")),
                             _stream(stream, q.device))
    if rc != GDN_OK:
        raise GdnError("gdn_bwd_noalloc", rc, lib)
    return out


def gdn_device_status() -> int:
    """Reads and clears the current device's status word: GDN_OK, or GDN_ERR_TIMEOUT when a
    kernel's bounded wait ran out since the last read (synchronises with the device)."""
    return load_library().gdn_device_status()


def gdn_debug_wait_probe(polls: int = 1000, stream=None) -> None:
    """Enqueue the timeout-path probe (include/gdn.h): one CTA whose bounded wait runs out after
    `polls` polls and records GDN_ERR_TIMEOUT in the device status word."""
    lib = load_library()
    rc = lib.gdn_debug_wait_probe(int(polls), _stream(stream))
    if rc != GDN_OK:
        raise GdnError("gdn_debug_wait_probe", rc, lib)


def gdn_diag_fma_tflops(packed: bool = False) -> float:
    """Measured FP32 FMA rate of the current device in TFLOP/s (include/gdn.h)."""
    lib = load_library()
    out = ctypes.c_double(0.0)
    rc = lib.gdn_diag_fma_tflops(1 if packed else 0, ctypes.byref(out))
    if rc != GDN_OK:
        raise GdnError("gdn_diag_fma_tflops", rc, lib)
    return out.value


def gdn_strerror(code: int) -> str:
    return load_library().gdn_strerror(code).decode()


def gdn_last_error() -> str:
    return load_library().gdn_last_error().decode()


def gdn_version() -> int:
    return load_library().gdn_version()


def _gate_shape(a, Hk, Dk, Dv):
    B, T, Hv = a.shape
    return make_shape(B, T, Hk, Hv, Dk, Dv, 64, _dtype_code(a))


def gdn_gates_fwd(a, b, A_log, dt_bias, *, Hk=None, Dk=32, Dv=4, stream=None):
    """g, beta = gdn_gates_fwd(a, b, A_log, dt_bias) on CUDA tensors (see include/gdn.h).
    a, b [B, T, Hv] (float32 or bfloat16); A_log, dt_bias [Hv] float32. Hk, Dk, Dv only
    complete the layer shape the library checks (defaults: Hk = Hv, Dk = 32, Dv = 4)."""
    torch = _torch()
    lib = load_library()
    B, T, Hv = a.shape
    _check("a", a, (B, T, Hv), a.dtype, a.device)
    _check("b", b, (B, T, Hv), a.dtype, a.device)
    _check("A_log", A_log, (Hv,), torch.float32, a.device)
    _check("dt_bias", dt_bias, (Hv,), torch.float32, a.device)
    _require_cuda(a)
    shape = _gate_shape(a, Hk or Hv, Dk, Dv)
    g = torch.empty_like(a)
    beta = torch.empty_like(a)
    rc = lib.gdn_gates_fwd(ctypes.byref(shape), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g),
                           _ptr(beta), _stream(stream, a.device))
    if rc != GDN_OK:
        raise GdnError("gdn_gates_fwd", rc, lib)
    return g, beta


def gdn_gates_bwd(a, b, A_log, dt_bias, dg, dbeta, *, Hk=None, Dk=32, Dv=4, stream=None):
    """dict(da, db, dA_log, ddt_bias) = gdn_gates_bwd(...) on CUDA tensors (see include/gdn.h)."""
    torch = _torch()
    lib = load_library()
    B, T, Hv = a.shape
    for name, t in (("a", a), ("b", b), ("dg", dg), ("dbeta", dbeta)):
        _check(name, t, (B, T, Hv), a.dtype, a.device)
    _check("A_log", A_log, (Hv,), torch.float32, a.device)
    _check("dt_bias", dt_bias, (Hv,), torch.float32, a.device)
    _require_cuda(a)
    shape = _gate_shape(a, Hk or Hv, Dk, Dv)
    out = {"da": torch.empty_like(a), "db": torch.empty_like(a),
           "dA_log": torch.empty_like(A_log), "ddt_bias": torch.empty_like(dt_bias)}
    rc = lib.gdn_gates_bwd(ctypes.byref(shape), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(dg),
                           _ptr(dbeta), _ptr(out["da"]), _ptr(out["db"]), _ptr(out["dA_log"]),
                           _ptr(out["ddt_bias"]), _stream(stream, a.device))
    if rc != GDN_OK:
        raise GdnError("gdn_gates_bwd", rc, lib)
    return out
