"""gdn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (for example code hosted by a runtime that owns all
device memory, or code that must not grow its device footprint after start-up), so they
cannot provide gdn_bwd's workspace. gdn_bwd_noalloc keeps that scratch in a fixed array
inside the library instead. These tests call it through the C ABI and check it against
gdn_bwd (the entry point with a caller workspace) on consecutive calls that share the
array, and check that problems beyond the array's size are refused up front.

This file is named so that pytest collects it last."""
import ctypes
import os

import pytest

import gdn_synthetic as gs
import gpu_harness as H
import oracle

torch = pytest.importorskip("torch")

SCRATCH_LIMIT = -7
NOALLOC_BYTES = 64 << 20   # GDN_BWD_NOALLOC_SCRATCH_BYTES in include/gdn.h


def _lib():
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return binding, binding.load_library()


def test_header_states_the_scratch_size():
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gdn.h")).read()
    assert "#define GDN_BWD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)" in text


def test_noalloc_refuses_problems_beyond_its_scratch():
    """Checked on the host before any CUDA call: the pointers below are never touched."""
    binding, lib = _lib()
    shape = binding.make_shape(1, 2048, 16, 64, 192, 128, 64, 1)
    assert lib.gdn_bwd_workspace_bytes(ctypes.byref(shape)) > NOALLOC_BYTES
    fake = ctypes.c_void_p(0x7F0000000000)
    rc = lib.gdn_bwd_noalloc(ctypes.byref(shape), *([fake] * 6), 1 << 40, fake, None, *([fake] * 5), None, None)
    assert rc == SCRATCH_LIMIT
    assert "GDN_BWD_NOALLOC_SCRATCH_BYTES" in lib.gdn_strerror(SCRATCH_LIMIT).decode()


def _noalloc(lib, binding, shape, t, ckpt, out):
    P = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gdn_bwd_noalloc(ctypes.byref(shape), P(t["q"]), P(t["k"]), P(t["v"]), P(t["g"]), P(t["beta"]),
                               P(ckpt), binding._room(ckpt), P(t["dy"]), P(t["dS_T"]), P(out["dq"]), P(out["dk"]),
                               P(out["dv"]), P(out["dg"]), P(out["dbeta"]), P(out["dS0"]), stream)


@pytest.mark.gpu
def test_noalloc_matches_gdn_bwd_on_consecutive_calls():
    """Both entry points run the same kernels on the same grid, so their results must agree
    bit for bit. The problems alternate between the two scratch layouts (the tensor-core
    backward's and the sequential backward's), so that every call after the first starts
    from scratch left dirty by a call of the other layout or of another shape."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding, lib = _lib()
    import gated_delta_rule_22_gb300 as gdn
    dev = torch.device("cuda:0")
    problems = [
        gs.Workload("na-tc", 1, 150, 1, 2, 128, 128, "bf16", "half", True, True, 64),     # tensor-core layout
        gs.Workload("na-f32", 2, 61, 2, 6, 64, 40, "f32", "strong", True, True, 16),      # sequential layout
        gs.Workload("na-f32", 2, 61, 2, 6, 64, 40, "f32", "strong", True, True, 16),      # same again
        gs.Workload("na-bf16", 1, 90, 1, 2, 128, 72, "bf16", "half", False, True, 32),    # sequential, bf16
        gs.Workload("na-tc2", 1, 200, 2, 4, 64, 64, "bf16", "strong", False, True, 64),   # tensor-core again
    ]
    for w in problems:
        inp = gs.make_inputs(w)
        t = H.to_device(inp, dev)
        shape = binding.make_shape(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, w.chunk, 0 if w.dtype == "f32" else 1)
        assert lib.gdn_bwd_workspace_bytes(ctypes.byref(shape)) <= NOALLOC_BYTES
        _, _, ckpt = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], chunk=w.chunk)
        ref = gdn.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ckpt, t["dy"], t["dS_T"], chunk=w.chunk)
        out = {n: torch.full_like(ref[n], float("nan")) for n in ref}
        rc = _noalloc(lib, binding, shape, t, ckpt, out)
        assert rc == 0, lib.gdn_strerror(rc).decode() + " " + lib.gdn_last_error().decode()
        torch.cuda.synchronize()
        for n in ref:
            assert torch.equal(out[n], ref[n]), (w.name, n)
        # and the pair is right: the oracle on the same inputs, at the parity tolerance
        want = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["dy"], inp["S0"], inp["dS_T"],
                          chunk=w.chunk)
        for n in ref:
            e = oracle.rel_l2(out[n].double().cpu().numpy(), want[n])
            assert e <= H.TOL[w.dtype], (w.name, n, e)
