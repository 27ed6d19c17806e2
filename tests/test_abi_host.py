"""The C-ABI library without a GPU: it loads, exports every function include/gdn.h
declares, sizes its buffers, and rejects bad arguments on the host before any CUDA call.

Pointers here are fake addresses that are never dereferenced: every call below returns
an error from the host-side checks, which run before anything is enqueued."""
import ctypes
import os

import pytest

from gated_delta_rule_22_gb300 import binding as B

OK, INVALID, MISALIGNED, UNSUPPORTED, WS_SMALL, CUDA, TIMEOUT = 0, -1, -2, -3, -4, -5, -6
FAKE = 0x7F0000000000  # 16-byte aligned, never touched


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return B.load_library()


def shape(**kw):
    base = dict(B=1, T=16, Hk=2, Hv=4, Dk=64, Dv=32, chunk=0, dtype=0)
    base.update(kw)
    return B.GdnShape(**base)


def _ck_bytes(lib, s, ck_bytes):
    if ck_bytes is None:
        ck_bytes = lib.gdn_ckpt_bytes(ctypes.byref(s)) if s is not None else 0
    return ck_bytes


def fwd(lib, s, ck_bytes=None, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, S0=None, y=FAKE, S_T=None, ckpt=FAKE)
    p.update(ptrs)
    args = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in
            ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt")]
    return lib.gdn_fwd(ctypes.byref(s) if s is not None else None, *args, _ck_bytes(lib, s, ck_bytes), None)


def bwd(lib, s, ws_bytes=None, ck_bytes=None, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, ckpt=FAKE, dy=FAKE, dS_T=None, dq=FAKE, dk=FAKE,
             dv=FAKE, dg=FAKE, dbeta=FAKE, dS0=None, ws=FAKE)
    p.update(ptrs)
    names = ("q", "k", "v", "g", "beta", "ckpt", "dy", "dS_T", "dq", "dk", "dv", "dg", "dbeta", "dS0", "ws")
    args = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in names]
    if ws_bytes is None:
        ws_bytes = lib.gdn_bwd_workspace_bytes(ctypes.byref(s)) if s is not None else 0
    return lib.gdn_bwd(ctypes.byref(s) if s is not None else None, *args[:6], _ck_bytes(lib, s, ck_bytes),
                       *args[6:], ws_bytes, None)


def test_exports_every_header_function(lib):
    names = B.header_functions()
    assert set(names) >= {"gdn_fwd", "gdn_bwd", "gdn_ckpt_bytes", "gdn_bwd_workspace_bytes",
                          "gdn_strerror", "gdn_last_error", "gdn_version"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/gdn.h but not exported"
    assert lib.gdn_version() == 2


def test_buffer_sizes_follow_the_plan(lib):
    """bf16 with chunk 64 and a supported Dk, Dv: the chunkwise form's saved buffer (larger than
    states + residuals) and workspace (dbeta and f partials per 32 value rows, and per 64-row block
    of a value head the [dY; dU], Delta and dS operand tiles; no dq, dk partials). When the chunked backward
    does not fit shared memory (Dk 128, Dv 256) the workspace is the sequential backward's
    (row-split partials), while the saved buffer stays chunkwise. Dv above 256 takes the
    sequential kernels altogether."""
    def sizes(**kw):
        s = shape(dtype=1, chunk=64, **kw)
        return lib.gdn_ckpt_bytes(ctypes.byref(s)), lib.gdn_bwd_workspace_bytes(ctypes.byref(s))
    # every supported (Dk, Dv) of the tensor-core forward, and whether its backward fits too
    table = {64: (64, 128, 192, 256), 128: (64, 128, 192), 192: (64, 128)}
    cases = [(Dk, Dv, Dv in table[Dk]) for Dk in (64, 128, 192) for Dv in (64, 128, 192, 256)]
    for Dk, Dv, chunked_bwd in cases:
        T, Hv = 150, 2
        ck, ws = sizes(T=T, Hk=1, Hv=Hv, Dk=Dk, Dv=Dv)
        NC = -(-T // 64)
        states, resid = Hv * NC * Dv * Dk * 4, T * Hv * Dv * 4
        assert ck > states + resid + 256, (Dk, Dv)
        row_split = 2 * T * Hv * (Dv // 64) * Dk * 4
        if chunked_bwd:
            r = lambda x: -(-x // 256) * 256  # noqa: E731
            ns = Dv // 64
            nblk = Hv * NC * ns
            want = (2 * r(T * Hv * ns * 2 * 4) + r(nblk * 128 * 64 * 2) + r(nblk * 64 * 64 * 2) + r(nblk * 64 * Dk * 2)
                    + r((Hv * NC + 1) * 4))   # the ready counters of the reverse sweep's chunks, the group counter
            assert ws == want, (Dk, Dv, ws, want)
        else:
            assert ws >= row_split, (Dk, Dv, ws)
    for Dk in (64, 128, 192):
        ck, _ = sizes(T=150, Hk=1, Hv=2, Dk=Dk, Dv=320)
        assert ck == (2 * 3 * 320 * Dk * 4 + 255) // 256 * 256 + 150 * 2 * 320 * 4
    # fp32 or another chunk size: the sequential layout, states + residuals exactly
    s = shape(dtype=1, chunk=32, T=150, Hk=1, Hv=2, Dk=128, Dv=128)
    assert lib.gdn_ckpt_bytes(ctypes.byref(s)) == (2 * 5 * 128 * 128 * 4 + 255) // 256 * 256 + 150 * 2 * 128 * 4


def test_checkpoint_bytes(lib):
    for T, C in ((16, 0), (37, 16), (1, 1), (128, 128), (2048, 64)):
        s = shape(T=T, chunk=C, Hv=6, Hk=3, Dk=96, Dv=20)
        nc = -(-T // (C or 64))
        states = -(-(1 * 6 * nc * 20 * 96 * 4) // 256) * 256   # chunk-start states, 256-byte rounded
        resid = 1 * T * 6 * 20 * 4                              # v - u per step and row
        assert lib.gdn_ckpt_bytes(ctypes.byref(s)) == states + resid
    assert lib.gdn_ckpt_bytes(ctypes.byref(shape(Hv=3))) == 0
    assert lib.gdn_ckpt_bytes(None) == 0


def test_workspace_bytes(lib):
    a = lib.gdn_bwd_workspace_bytes(ctypes.byref(shape(T=16)))
    b = lib.gdn_bwd_workspace_bytes(ctypes.byref(shape(T=1024)))
    assert 0 < a < b and a % 256 == 0 and b % 256 == 0
    assert lib.gdn_bwd_workspace_bytes(ctypes.byref(shape(Dk=40))) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), INVALID), (dict(B=-1), INVALID), (dict(Dv=0), INVALID), (dict(dtype=7), INVALID),
    (dict(chunk=-1), INVALID), (dict(Hv=3), UNSUPPORTED), (dict(Dk=48), UNSUPPORTED),
    (dict(Dk=288), UNSUPPORTED), (dict(Dv=6), UNSUPPORTED), (dict(Dv=4100), UNSUPPORTED),
    (dict(chunk=129), UNSUPPORTED), (dict(Hv=70000, Hk=1), UNSUPPORTED),
])
def test_bad_shapes_rejected(lib, kw, code):
    s = shape(**kw)
    assert fwd(lib, s) == code
    assert bwd(lib, s, ws_bytes=1 << 40) == code


def test_null_shape_and_pointers(lib):
    assert fwd(lib, None) == INVALID
    assert bwd(lib, None, ws_bytes=0) == INVALID
    s = shape()
    for n in ("q", "k", "v", "g", "beta", "y"):
        assert fwd(lib, s, **{n: None}) == INVALID, n
    # the forward may run without a saved-for-backward buffer (inference / decode): a null
    # ckpt passes the argument checks (shown here by the next check, alignment, firing)
    assert fwd(lib, s, ckpt=None, q=FAKE + 4) == MISALIGNED
    for n in ("q", "k", "v", "g", "beta", "ckpt", "dy", "dq", "dk", "dv", "dg", "dbeta", "ws"):
        assert bwd(lib, s, **{n: None}) == INVALID, n


def test_misaligned_pointers(lib):
    s = shape()
    for n in ("q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt"):
        assert fwd(lib, s, **{n: FAKE + 4}) == MISALIGNED, n
    for n in ("q", "dS_T", "dq", "dS0", "ws"):
        assert bwd(lib, s, **{n: FAKE + 8}) == MISALIGNED, n


def test_workspace_too_small(lib):
    s = shape()
    need = lib.gdn_bwd_workspace_bytes(ctypes.byref(s))
    assert bwd(lib, s, ws_bytes=need - 1) == WS_SMALL
    assert bwd(lib, s, ws_bytes=0) == WS_SMALL


@pytest.mark.parametrize("kw", [dict(), dict(dtype=1, chunk=64, T=150, Hk=1, Hv=2, Dk=192, Dv=128)])
def test_checkpoint_buffer_too_small(lib, kw):
    """A saved-for-backward buffer sized from the [B, Hv, NC, Dv, Dk] states alone (or one byte
    short of gdn_ckpt_bytes) is refused on the host, before anything is enqueued, by both the
    forward and the backward (the fake pointers are never touched). The tensor-core shape's
    buffer holds more than the states, so the states-only size is short there too."""
    s = shape(**kw)
    need = lib.gdn_ckpt_bytes(ctypes.byref(s))
    NC = -(-s.T // (s.chunk or 64))
    states = s.B * s.Hv * NC * s.Dv * s.Dk * 4
    assert states < need
    for n in (need - 1, states, 0):
        assert fwd(lib, s, ck_bytes=n) == WS_SMALL, n
        assert bwd(lib, s, ck_bytes=n) == WS_SMALL, n
        fake = ctypes.c_void_p(FAKE)
        rc = lib.gdn_bwd_noalloc(ctypes.byref(s), *([fake] * 6), n, fake, None, *([fake] * 5), None, None)
        assert rc == WS_SMALL or rc == -7, n   # or refused for its scratch size first
    # no saved buffer (inference): its size is not looked at
    assert fwd(lib, s, ck_bytes=0, ckpt=None, q=FAKE + 4) == MISALIGNED


GATE_FWD = ("a", "b", "A_log", "dt_bias", "g", "beta")
GATE_BWD = ("a", "b", "A_log", "dt_bias", "dg", "dbeta", "da", "db", "dA_log", "ddt_bias")


def gates(lib, s, names, **ptrs):
    p = {n: FAKE for n in names}
    p.update(ptrs)
    args = [ctypes.c_void_p(p[n]) if p[n] is not None else None for n in names]
    f = lib.gdn_gates_fwd if names == GATE_FWD else lib.gdn_gates_bwd
    return f(ctypes.byref(s) if s is not None else None, *args, None)


def test_gate_argument_checks(lib):
    s = shape()
    for names in (GATE_FWD, GATE_BWD):
        assert gates(lib, None, names) == INVALID
        assert gates(lib, shape(Hv=3), names) == UNSUPPORTED        # Hv % Hk
        assert gates(lib, shape(B=65535, T=40000), names) == UNSUPPORTED   # B*T >= 2^31
        for n in names:
            assert gates(lib, s, names, **{n: None}) == INVALID, n
            assert gates(lib, s, names, **{n: FAKE + 4}) == MISALIGNED, n


def test_error_strings(lib):
    texts = {c: lib.gdn_strerror(c).decode() for c in (OK, INVALID, MISALIGNED, UNSUPPORTED, WS_SMALL, CUDA, TIMEOUT)}
    assert len(set(texts.values())) == len(texts)
    assert "unknown" in lib.gdn_strerror(42).decode()
    assert lib.gdn_last_error().decode() == ""


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        B.load_library(str(tmp_path / "libgdn.so"))


def test_binding_has_every_header_function(lib):
    import gated_delta_rule_22_gb300 as gdn
    missing = [f for f in B.header_functions() if not callable(getattr(gdn, f, None))]
    assert not missing, missing


def _host_tensors(dtype=None):
    import torch
    import gdn_synthetic as gs
    w = gs.WORKLOADS["tiny"]
    inp = gs.make_inputs(w)
    dt = dtype or torch.float32
    return w, {n: torch.from_numpy(inp[n]).to(dt) for n in ("q", "k", "v", "g", "beta", "dy")}


def test_binding_refuses_host_tensors(lib):
    """The C ABI takes device pointers; the binding stops host tensors before the call."""
    import gated_delta_rule_22_gb300 as gdn
    _, t = _host_tensors()
    with pytest.raises(ValueError, match="CUDA tensors"):
        gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"])
    ck = gdn.new_ckpt(t["q"], t["v"])
    for fn in (gdn.gdn_bwd, gdn.gdn_bwd_noalloc):
        with pytest.raises(ValueError, match="CUDA tensors"):
            fn(t["q"], t["k"], t["v"], t["g"], t["beta"], ck, t["dy"])
    import torch
    Hv = t["g"].shape[2]
    A_log, dt_bias = torch.zeros(Hv), torch.zeros(Hv)
    with pytest.raises(ValueError, match="CUDA tensors"):
        gdn.gdn_gates_fwd(t["g"], t["beta"], A_log, dt_bias)
    with pytest.raises(ValueError, match="CUDA tensors"):
        gdn.gdn_gates_bwd(t["g"], t["beta"], A_log, dt_bias, t["g"], t["beta"])


def test_binding_checks_caller_outputs(lib):
    """Output tensors a caller passes in are checked like the inputs (shape, dtype, layout),
    so a wrong one cannot reach a kernel as a too-small buffer."""
    import torch
    import gated_delta_rule_22_gb300 as gdn
    _, t = _host_tensors()
    q, k, v, g, beta, dy = (t[n] for n in ("q", "k", "v", "g", "beta", "dy"))
    with pytest.raises(ValueError, match="y has shape"):
        gdn.gdn_fwd(q, k, v, g, beta, y=torch.empty(v.shape[0], v.shape[1] - 1, *v.shape[2:]))
    with pytest.raises(ValueError, match="S_T has shape"):
        gdn.gdn_fwd(q, k, v, g, beta, S_T=torch.empty(1))
    with pytest.raises(ValueError, match="ckpt"):
        gdn.gdn_fwd(q, k, v, g, beta, ckpt=torch.empty(1))
    ck = gdn.new_ckpt(q, v)
    good = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
            "dg": torch.empty_like(g), "dbeta": torch.empty_like(beta)}
    with pytest.raises(ValueError, match="out lacks dv"):
        gdn.gdn_bwd(q, k, v, g, beta, ck, dy, out={n: x for n, x in good.items() if n != "dv"})
    with pytest.raises(TypeError, match="dq has dtype"):
        gdn.gdn_bwd(q, k, v, g, beta, ck, dy, out=dict(good, dq=torch.empty_like(q, dtype=torch.float64)))
    with pytest.raises(ValueError, match="dk must be contiguous"):
        gdn.gdn_bwd(q, k, v, g, beta, ck, dy, out=dict(good, dk=torch.empty_like(k).transpose(2, 3)
                                                       .contiguous().transpose(2, 3)))
    with pytest.raises(ValueError, match="dS0 has shape"):
        gdn.gdn_bwd_noalloc(q, k, v, g, beta, ck, dy, out=dict(good, dS0=torch.empty(3)))
    with pytest.raises(ValueError, match="workspace must be"):
        gdn.gdn_bwd(q, k, v, g, beta, ck, dy, workspace=torch.empty(64, dtype=torch.uint8)[::2])
    # all of it well formed: only the device is wrong
    with pytest.raises(ValueError, match="CUDA tensors"):
        gdn.gdn_bwd(q, k, v, g, beta, ck, dy, out=good, workspace=torch.empty(64, dtype=torch.uint8))


def test_diagnostic_argument_checks(lib):
    """Refused on the host before any CUDA call."""
    assert lib.gdn_debug_wait_probe(0, None) == INVALID
    assert lib.gdn_debug_wait_probe((1 << 24) + 1, None) == INVALID
    assert lib.gdn_diag_fma_tflops(0, None) == INVALID
