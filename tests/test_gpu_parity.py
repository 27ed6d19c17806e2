"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle on the same
seeded inputs, element by element via relative L2 per output tensor.

Tolerances: 1e-5 for float32 inputs (every output, dg under strong decay included) and
5e-3 for bf16 inputs against the oracle run on the bf16-rounded values."""
import ctypes
import os

import numpy as np
import pytest

import gdn_synthetic as gs
import gpu_harness as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return torch.device("cuda:0")


def check(errs, tol, label):
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"{label}: outputs above tolerance {tol:g}: {bad} (all: {errs})"


# ---------------------------------------------------------------- whole-tensor parity
# Every named workload at its full size, every output compared whole (the oracle runs on all
# host cores: about a minute in all, most of it the T = 32768 workload).
@pytest.mark.parametrize("name", ["tiny", "stress-strong", "stress-weak", "linattn-T256", "linattn-T512",
                                  "linattn-T1024", "linattn-T2048", "batched", "long"])
def test_parity_full(dev, name):
    w = gs.WORKLOADS[name]
    inp = gs.make_inputs(w)
    out = H.run_gpu(inp, dev)
    got = H.to_numpy(out)
    del out
    torch.cuda.empty_cache()
    ref = H.run_oracle(inp)
    errs = H.errors(got, ref)
    print(name, {n: f"{e:.2e}" for n, e in errs.items()})
    H.log_errors(name, errs)
    check(errs, H.TOL[w.dtype], name)


EDGE = [
    gs.Workload("T1-Dv4", 1, 1, 1, 1, 32, 4, "f32", "weak", True, True, 64),
    gs.Workload("ragged-T-gqa3", 2, 37, 2, 6, 64, 24, "f32", "strong", True, True, 16),
    gs.Workload("Dv100-C7-Dk96", 1, 50, 1, 2, 96, 100, "f32", "weak", False, True, 7),
    gs.Workload("C1-Dk160", 1, 20, 2, 2, 160, 12, "f32", "strong", True, False, 1),
    gs.Workload("C128-gt-T-Dk224", 1, 40, 1, 3, 224, 8, "f32", "weak", False, False, 128),
    gs.Workload("Dk256-C128-Dv132", 1, 300, 1, 1, 256, 132, "f32", "strong", True, True, 128),
    gs.Workload("bf16-ragged-half", 2, 45, 2, 4, 128, 36, "bf16", "half", True, True, 32),
    gs.Workload("bf16-strong-Dk192", 1, 70, 1, 4, 192, 128, "bf16", "strong", False, False, 64),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_parity_edge_cases(dev, w):
    inp = gs.make_inputs(w)
    got = H.to_numpy(H.run_gpu(inp, dev))
    ref = H.run_oracle(inp)
    errs = H.errors(got, ref)
    print(w.name, {n: f"{e:.2e}" for n, e in errs.items()})
    check(errs, H.TOL[w.dtype], w.name)


# ------------------------------------------------------------------- structural checks
def _bitwise_equal(a: dict, b: dict):
    for n in a:
        if a[n] is not None:
            assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("name", ["linattn-T256", "linattn-T2048", "batched"])
def test_deterministic_across_runs(dev, name):
    inp = gs.make_inputs(gs.WORKLOADS[name])
    a = H.run_gpu(inp, dev)
    b = H.run_gpu(inp, dev)
    _bitwise_equal(a, b)


# B = 3 on the sequential kernels (fp32); B = 8 on the tensor-core kernels (bf16, 2 kv heads x
# 16 chunks x 8 rows = 256 groups of value heads: more than a GB300 has SMs, so the gradient
# kernel's CTAs take one or two groups each, at other offsets than in the B = 1 runs)
@pytest.mark.parametrize("w", [gs.Workload("b3", 3, 29, 2, 4, 64, 40, "f32", "half", True, True, 8),
                               gs.Workload("b8-tc", 8, 1000, 2, 8, 128, 128, "bf16", "half", True, True, 64)],
                         ids=lambda w: w.name)
def test_batch_rows_independent(dev, w):
    """Batch row b of a B-row problem gives, bit for bit, what the one-row problem of its
    inputs gives: nothing in any reduction depends on the other rows or on where the grid
    cuts the work."""
    inp = gs.make_inputs(w)
    full = H.run_gpu(inp, dev)
    for b in range(w.B):
        one = {n: (x[b:b + 1] if isinstance(x, np.ndarray) else x) for n, x in inp.items()}
        one["workload"] = gs.Workload(**{**w.as_dict(), "B": 1})
        part = H.run_gpu(one, dev)
        for n in H.OUTPUTS:
            assert torch.equal(full[n][b:b + 1], part[n]), (b, n)


def test_optional_states(dev):
    import gated_delta_rule_22_gb300 as gdn
    w = gs.Workload("opt", 1, 33, 2, 4, 64, 16, "f32", "weak", False, False, 16)
    inp = gs.make_inputs(w)
    t = H.to_device(inp, dev)
    zeros = torch.zeros((1, 4, 16, 64), dtype=torch.float32, device=dev)
    y0, S0_T, ck0 = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], None, chunk=16)
    y1, S1_T, ck1 = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], zeros, chunk=16)
    y2, S2_T, ck2 = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], None, chunk=16, want_S_T=False)
    assert S2_T is None
    for a, b in ((y0, y1), (y0, y2), (S0_T, S1_T), (ck0, ck1), (ck0, ck2)):
        assert torch.equal(a, b)
    g0 = gdn.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ck0, t["dy"], None, chunk=16)
    g1 = gdn.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ck0, t["dy"], zeros, chunk=16)
    g2 = gdn.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ck0, t["dy"], None, chunk=16, want_dS0=False)
    assert g2["dS0"] is None
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(g0[n], g1[n]) and torch.equal(g0[n], g2[n]), n
    assert torch.equal(g0["dS0"], g1["dS0"])


def test_chunk_size_changes_only_checkpoints(dev):
    """y and S_T do not depend on the checkpoint interval at all (bitwise); the gradients
    depend on it only through float32 rounding inside the re-computation."""
    base = gs.Workload("cs", 1, 70, 2, 4, 128, 32, "f32", "strong", True, True, 64)
    ref = None
    for C in (1, 5, 16, 64, 128):
        out = H.run_gpu(gs.make_inputs(base, chunk=C), dev)
        if ref is None:
            ref = out
            continue
        assert torch.equal(out["y"], ref["y"]) and torch.equal(out["S_T"], ref["S_T"]), C
        for n in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
            e = float((out[n].double() - ref[n].double()).norm() / ref[n].double().norm())
            assert e < 1e-5, (C, n, e)


def test_device_side_argument_errors(dev):
    import gated_delta_rule_22_gb300 as gdn
    from gated_delta_rule_22_gb300 import binding as B
    w = gs.Workload("err", 1, 8, 1, 1, 32, 8, "f32", "weak")
    t = H.to_device(gs.make_inputs(w), dev)
    y, _, ck = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"])
    shape = B.make_shape(1, 8, 1, 1, 32, 8, 64, 0)
    need = gdn.gdn_bwd_workspace_bytes(shape)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ck, t["dy"],
                    workspace=torch.empty(need - 256, dtype=torch.uint8, device=dev))
    assert ei.value.code == -4
    lib = B.load_library()
    P = lambda x, off=0: ctypes.c_void_p(x.data_ptr() + off)  # noqa: E731
    rc = lib.gdn_fwd(ctypes.byref(shape), P(t["q"], 4), P(t["k"]), P(t["v"]), P(t["g"]), P(t["beta"]),
                     None, P(y), None, P(ck), gdn.gdn_ckpt_bytes(shape), None)
    assert rc == -2
    # a saved-for-backward buffer one byte short, or sized from the states alone
    for n in (gdn.gdn_ckpt_bytes(shape) - 1, ck.numel() * 4):
        rc = lib.gdn_fwd(ctypes.byref(shape), P(t["q"]), P(t["k"]), P(t["v"]), P(t["g"]), P(t["beta"]),
                         None, P(y), None, P(ck), n, None)
        assert rc == -4, n
