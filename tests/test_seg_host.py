"""The sequence-parallel entry points without a GPU: the sizes they ask for, and their host-side
argument checks (fake, never-dereferenced pointers; every call below returns an error before
anything is enqueued)."""
import ctypes
import os

import pytest

from gated_delta_rule_22_gb300 import binding as B

OK, INVALID, MISALIGNED, UNSUPPORTED, SMALL = 0, -1, -2, -3, -4
FAKE = 0x7F0000000000


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return B.load_library()


def shape(**kw):
    base = dict(B=2, T=512, Hk=2, Hv=4, Dk=128, Dv=128, chunk=64, dtype=1)
    base.update(kw)
    return B.GdnShape(**base)


def r256(x):
    return -(-x // 256) * 256


def test_sizes_are_those_of_the_viewed_problem(lib):
    """Segments of whole chunks: the saved buffer is the viewed problem's (B * P rows of T / P
    steps) followed by the maps and their transposes; the workspace is two state arrays and the
    viewed backward's."""
    for P in (1, 2, 4, 8):
        s = shape()
        v = shape(B=2 * P, T=512 // P)
        maps = 2 * (2 * P * 4 * 128 * 128 * 4)           # the maps and their transposes
        states = 2 * P * 4 * 128 * 128 * 4
        assert lib.gdn_seg_ckpt_bytes(ctypes.byref(s), P) == r256(lib.gdn_ckpt_bytes(ctypes.byref(v))) + r256(maps)
        assert lib.gdn_seg_workspace_bytes(ctypes.byref(s), P) == (
            2 * r256(states) + lib.gdn_bwd_workspace_bytes(ctypes.byref(v)))
        # the viewed problem's saved buffer is as large as the whole problem's
        assert lib.gdn_ckpt_bytes(ctypes.byref(v)) == lib.gdn_ckpt_bytes(ctypes.byref(s))


@pytest.mark.parametrize("kw,P", [
    (dict(), 0), (dict(), -1), (dict(), 3),            # 512 is not a multiple of 64 * 3
    (dict(T=500), 1),                                  # a ragged last chunk
    (dict(dtype=0), 2),                                # fp32: the sequential kernels
    (dict(chunk=32), 2),                               # another checkpoint interval
    (dict(Dk=96), 2),                                  # a Dk the tensor-core kernels do not take
    (dict(Dk=128, Dv=256), 2),                         # the tensor-core backward does not fit
])
def test_shapes_it_does_not_take(lib, kw, P):
    s = shape(**kw)
    assert lib.gdn_seg_ckpt_bytes(ctypes.byref(s), P) == 0
    assert lib.gdn_seg_workspace_bytes(ctypes.byref(s), P) == 0
    f = ctypes.c_void_p(FAKE)
    rc = lib.gdn_fwd_seg(ctypes.byref(s), P, f, f, f, f, f, None, f, None, f, 1 << 40, f, 1 << 40, None)
    assert rc in (UNSUPPORTED, INVALID), rc


def seg_fwd(lib, s, P, ck=None, ws=None, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, S0=None, y=FAKE, S_T=None, ckpt=FAKE, work=FAKE)
    p.update(ptrs)
    a = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in
         ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt", "work")]
    ck = lib.gdn_seg_ckpt_bytes(ctypes.byref(s), P) if ck is None else ck
    ws = lib.gdn_seg_workspace_bytes(ctypes.byref(s), P) if ws is None else ws
    return lib.gdn_fwd_seg(ctypes.byref(s), P, *a[:9], ck, a[9], ws, None)


def seg_bwd(lib, s, P, ck=None, ws=None, **ptrs):
    names = ("q", "k", "v", "g", "beta", "ckpt", "dy", "dS_T", "dq", "dk", "dv", "dg", "dbeta", "dS0", "work")
    p = {n: FAKE for n in names}
    p.update(dS_T=None, dS0=None)
    p.update(ptrs)
    a = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in names]
    ck = lib.gdn_seg_ckpt_bytes(ctypes.byref(s), P) if ck is None else ck
    ws = lib.gdn_seg_workspace_bytes(ctypes.byref(s), P) if ws is None else ws
    return lib.gdn_bwd_seg(ctypes.byref(s), P, *a[:6], ck, *a[6:], ws, None)


def test_argument_checks(lib):
    s, P = shape(), 4
    need_ck = lib.gdn_seg_ckpt_bytes(ctypes.byref(s), P)
    need_ws = lib.gdn_seg_workspace_bytes(ctypes.byref(s), P)
    for call in (seg_fwd, seg_bwd):
        assert call(lib, s, P, ck=need_ck - 1) == SMALL
        assert call(lib, s, P, ws=need_ws - 1) == SMALL
        assert call(lib, s, P, q=FAKE + 8) == MISALIGNED
        assert call(lib, s, P, q=None) == INVALID
        assert call(lib, s, P, ckpt=None) == INVALID
        assert call(lib, s, P, work=None) == INVALID
    assert seg_fwd(lib, s, P, y=None) == INVALID
    assert seg_bwd(lib, s, P, dy=None) == INVALID
    assert lib.gdn_fwd_seg(None, P, *([None] * 9), 0, None, 0, None) == INVALID


def test_segment_count_fills_the_gpu(lib):
    """The chosen count fills 152 SMs with the sweeps' grid and no more: the long workload's
    8-way head split takes 8 segments, a 4-head Dk = Dv = 128 case 16, and the layer with all 64
    value heads (128 sweep CTAs already) none."""
    tp8 = B.GdnShape(B=1, T=32768, Hk=2, Hv=8, Dk=192, Dv=128, chunk=64, dtype=1)
    h4 = B.GdnShape(B=1, T=32768, Hk=4, Hv=4, Dk=128, Dv=128, chunk=64, dtype=1)
    full = B.GdnShape(B=1, T=32768, Hk=16, Hv=64, Dk=192, Dv=128, chunk=64, dtype=1)
    assert lib.gdn_seg_choose(ctypes.byref(tp8), 152) == 8
    assert lib.gdn_seg_choose(ctypes.byref(h4), 152) == 16
    assert lib.gdn_seg_choose(ctypes.byref(full), 152) == 1
    # T limits the count: 128 steps hold two chunks
    short = B.GdnShape(B=1, T=128, Hk=2, Hv=8, Dk=192, Dv=128, chunk=64, dtype=1)
    assert lib.gdn_seg_choose(ctypes.byref(short), 152) == 2
    # shapes the tensor-core kernels do not take, and nonsense SM counts: the plain calls
    assert lib.gdn_seg_choose(ctypes.byref(shape(dtype=0)), 152) == 1
    assert lib.gdn_seg_choose(ctypes.byref(tp8), 0) == 1
    assert lib.gdn_seg_choose(None, 152) == 1
