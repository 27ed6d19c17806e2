"""The re-computation mode's entry points without a GPU: the sizes they ask for (the saved buffer
is the checkpoints and residuals only) and their host-side argument checks (fake,
never-dereferenced pointers; every call below returns an error before anything is enqueued)."""
import ctypes
import os

import pytest

from gated_delta_rule_22_gb300 import binding as B

INVALID, MISALIGNED, UNSUPPORTED, SMALL = -1, -2, -3, -4
FAKE = 0x7F0000000000


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return B.load_library()


def shape(**kw):
    base = dict(B=2, T=500, Hk=2, Hv=4, Dk=192, Dv=128, chunk=64, dtype=1)
    base.update(kw)
    return B.GdnShape(**base)


def r256(x):
    return -(-x // 256) * 256


def test_saved_buffer_is_checkpoints_and_residuals(lib):
    for kw in (dict(), dict(T=64, Dk=64, Dv=64), dict(B=1, T=2048, Hk=16, Hv=64)):
        s = shape(**kw)
        NC = -(-s.T // 64)
        states = r256(s.B * s.Hv * NC * s.Dv * s.Dk * 4)
        resid = s.B * s.T * s.Hv * s.Dv * 4
        assert lib.gdn_rc_ckpt_bytes(ctypes.byref(s)) == states + r256(resid)
        full = lib.gdn_ckpt_bytes(ctypes.byref(s))
        prod = lib.gdn_rc_fwd_workspace_bytes(ctypes.byref(s))
        # the products moved out of the saved buffer into the workspace
        assert states + r256(resid) + prod == full
        assert lib.gdn_rc_bwd_workspace_bytes(ctypes.byref(s)) == prod + lib.gdn_bwd_workspace_bytes(ctypes.byref(s))


@pytest.mark.parametrize("kw", [dict(dtype=0), dict(chunk=32), dict(Dk=96), dict(Dk=128, Dv=256)])
def test_shapes_it_does_not_take(lib, kw):
    s = shape(**kw)
    assert lib.gdn_rc_ckpt_bytes(ctypes.byref(s)) == 0
    assert lib.gdn_rc_fwd_workspace_bytes(ctypes.byref(s)) == 0
    assert lib.gdn_rc_bwd_workspace_bytes(ctypes.byref(s)) == 0
    f = ctypes.c_void_p(FAKE)
    assert lib.gdn_fwd_rc(ctypes.byref(s), f, f, f, f, f, None, f, None, f, 1 << 40, f, 1 << 40, None) == UNSUPPORTED


def rc_fwd(lib, s, ck=None, ws=None, **ptrs):
    names = ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt", "work")
    p = {n: FAKE for n in names}
    p.update(S0=None, S_T=None)
    p.update(ptrs)
    a = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in names]
    ck = lib.gdn_rc_ckpt_bytes(ctypes.byref(s)) if ck is None else ck
    ws = lib.gdn_rc_fwd_workspace_bytes(ctypes.byref(s)) if ws is None else ws
    return lib.gdn_fwd_rc(ctypes.byref(s), *a[:9], ck, a[9], ws, None)


def rc_bwd(lib, s, ck=None, ws=None, **ptrs):
    names = ("q", "k", "v", "g", "beta", "ckpt", "dy", "dS_T", "dq", "dk", "dv", "dg", "dbeta", "dS0", "work")
    p = {n: FAKE for n in names}
    p.update(dS_T=None, dS0=None)
    p.update(ptrs)
    a = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in names]
    ck = lib.gdn_rc_ckpt_bytes(ctypes.byref(s)) if ck is None else ck
    ws = lib.gdn_rc_bwd_workspace_bytes(ctypes.byref(s)) if ws is None else ws
    return lib.gdn_bwd_rc(ctypes.byref(s), *a[:6], ck, *a[6:], ws, None)


def test_argument_checks(lib):
    s = shape()
    for call, ws_q in ((rc_fwd, lib.gdn_rc_fwd_workspace_bytes), (rc_bwd, lib.gdn_rc_bwd_workspace_bytes)):
        assert call(lib, s, ck=lib.gdn_rc_ckpt_bytes(ctypes.byref(s)) - 1) == SMALL
        assert call(lib, s, ws=ws_q(ctypes.byref(s)) - 1) == SMALL
        assert call(lib, s, k=FAKE + 4) == MISALIGNED
        assert call(lib, s, q=None) == INVALID
        assert call(lib, s, ckpt=None) == INVALID
        assert call(lib, s, work=None) == INVALID
    assert rc_fwd(lib, s, y=None) == INVALID
    assert rc_bwd(lib, s, dy=None) == INVALID
    assert lib.gdn_fwd_rc(None, *([None] * 9), 0, None, 0, None) == INVALID
    assert lib.gdn_bwd_rc(None, *([None] * 6), 0, *([None] * 9), 0, None) == INVALID


def test_inference_forward_sizes_and_checks(lib):
    """gdn_fwd_infer: its workspace is the per-chunk products only; it takes the shapes the
    chunkwise forward takes (including value widths the chunkwise backward does not)."""
    s = shape()
    assert lib.gdn_infer_workspace_bytes(ctypes.byref(s)) == lib.gdn_rc_fwd_workspace_bytes(ctypes.byref(s))
    wide = shape(Dk=128, Dv=256)
    assert lib.gdn_infer_workspace_bytes(ctypes.byref(wide)) > 0
    for kw in (dict(dtype=0), dict(chunk=32), dict(Dk=96)):
        bad = shape(**kw)
        assert lib.gdn_infer_workspace_bytes(ctypes.byref(bad)) == 0
    f = ctypes.c_void_p(FAKE)
    need = lib.gdn_infer_workspace_bytes(ctypes.byref(s))

    def call(sh=s, ws=need, **ptrs):
        names = ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "work")
        p = {n: FAKE for n in names}
        p.update(S0=None, S_T=None)
        p.update(ptrs)
        a = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in names]
        return lib.gdn_fwd_infer(ctypes.byref(sh), *a[:8], a[8], ws, None)

    assert call(sh=shape(dtype=0)) == UNSUPPORTED
    assert call(ws=need - 1) == SMALL
    assert call(v=FAKE + 8) == MISALIGNED
    assert call(y=None) == INVALID
    assert call(work=None) == INVALID
    assert lib.gdn_fwd_infer(None, f, f, f, f, f, None, f, None, f, need, None) == INVALID
