"""GPU parity of the sequence-parallel form through the C ABI (gdn_fwd_seg / gdn_bwd_seg): the
sequence is cut into P segments of whole chunks, each segment's affine state map is taken on
the tensor cores, a scan over the segments gives every segment's start state (and, backwards,
its end adjoint), and the chunkwise kernels run on the B * P segment rows.

Checked against the float64 oracle run on the WHOLE sequence (no segments): y, S_T, the
chunk-start checkpoints (the segment rows' checkpoints put back in [B, Hv, NC, Dv, Dk] order)
and every gradient, with start states and final-state cotangents, GQA, every supported key
width, 2 to 16 segments, one chunk per segment, and the long-context workloads at full size
(two kv-head groups compared). One segment gives the plain chunkwise call's outputs bit for bit, and two
runs agree bit for bit. Tolerance 5e-3 relative L2 (bf16 inputs)."""
import os

import numpy as np
import pytest

import gdn_synthetic as gs
import gpu_harness as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return torch.device("cuda:0")


def run_seg(inp, P, dev):
    """Both sequence-parallel calls; the checkpoints returned as the [B, Hv, NC, Dv, Dk] tensor
    of the whole problem."""
    import gated_delta_rule_22_gb300 as gdn
    w = inp["workload"]
    t = H.to_device(inp, dev)
    y, S_T, ck = gdn.gdn_fwd_seg(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], segments=P)
    gr = gdn.gdn_bwd_seg(t["q"], t["k"], t["v"], t["g"], t["beta"], ck, t["dy"], t["dS_T"], segments=P)
    torch.cuda.synchronize()
    NC = w.T // 64
    n = w.B * w.Hv * NC * w.Dv * w.Dk
    states = ck[:4 * n].view(torch.float32).reshape(w.B, P, w.Hv, NC // P, w.Dv, w.Dk)
    ckpt = states.permute(0, 2, 1, 3, 4, 5).reshape(w.B, w.Hv, NC, w.Dv, w.Dk)
    return {"y": y, "S_T": S_T, "ckpt": ckpt, **gr}


CASES = [
    # (workload, segments)
    (gs.Workload("seg-few-heads", 1, 1024, 1, 2, 128, 128, "bf16", "weak", True, True, 64), 4),
    (gs.Workload("seg-gqa-Dk192-one-chunk", 2, 512, 2, 4, 192, 128, "bf16", "strong", True, True, 64), 8),
    (gs.Workload("seg-Dk64-Dv192-P3", 1, 768, 1, 3, 64, 192, "bf16", "half", True, False, 64), 3),
    (gs.Workload("seg-P16", 1, 2048, 1, 2, 128, 64, "bf16", "weak", False, True, 64), 16),
    (gs.Workload("seg-P2-noS0", 2, 256, 2, 2, 128, 128, "bf16", "half", False, False, 64), 2),
]


@pytest.mark.parametrize("w,P", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_segmented_parity(dev, w, P):
    inp = gs.make_inputs(w)
    got = H.to_numpy(run_seg(inp, P, dev))
    ref = H.run_oracle(inp)
    errs = H.errors(got, ref)
    print(w.name, P, {n: f"{e:.2e}" for n, e in errs.items()})
    H.log_errors(f"{w.name}-P{P}", errs)
    assert set(errs) == set(H.OUTPUTS), errs
    bad = {n: e for n, e in errs.items() if not e <= H.TOL["bf16"]}
    assert not bad, (w.name, P, bad)


def test_degenerate_gates_at_segment_edges(dev):
    """g = 0 (the state wiped) and beta = 0 at the first and last steps of segments: a map that
    is exactly zero, and segments whose first or last step writes nothing."""
    w = gs.Workload("seg-degenerate", 1, 512, 1, 2, 128, 64, "bf16", "weak", True, True, 64)
    inp = gs.make_inputs(w)
    g, beta = inp["g"].copy(), inp["beta"].copy()
    g[0, [0, 127, 128, 300, 511], :] = 0.0
    beta[0, [128, 255, 256, 383], :] = 0.0
    inp["g"], inp["beta"] = g, beta
    got = H.to_numpy(run_seg(inp, 4, dev))
    errs = H.errors(got, H.run_oracle(inp))
    print(errs)
    bad = {n: e for n, e in errs.items() if not e <= H.TOL["bf16"]}
    assert not bad, bad


def test_one_segment_is_the_plain_call(dev):
    w = gs.Workload("seg-P1", 1, 320, 2, 4, 128, 128, "bf16", "half", True, True, 64)
    inp = gs.make_inputs(w)
    a = run_seg(inp, 1, dev)
    b = H.run_gpu(inp, dev)
    for n in H.OUTPUTS:
        assert torch.equal(a[n], b[n]), n


def test_segmented_is_deterministic(dev):
    w, P = CASES[1]
    inp = gs.make_inputs(w)
    a = run_seg(inp, P, dev)
    b = run_seg(inp, P, dev)
    for n in H.OUTPUTS:
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("name,P", [("long", 4), ("long-tp8", 8)])
def test_segmented_long_context(dev, name, P):
    """The long-context workloads at full size, in the segment counts the benchmark times: T =
    32768, Dk = 192 (64 value heads on 16 kv heads in 4 segments; the 8-way head split, 8 value
    heads on 2 kv heads, in 8): the first and last kv-head groups of every output against the
    oracle on those groups."""
    w = gs.WORKLOADS[name]
    inp = gs.make_inputs(w)
    out = run_seg(inp, P, dev)
    for hk in (0, w.Hk - 1):
        got = H.group_outputs(out, w, 0, hk)
        ref = H.oracle_group(inp, 0, hk)
        errs = H.errors(got, ref)
        print(name, "P", P, "group", hk, {n: f"{e:.2e}" for n, e in errs.items()})
        H.log_errors(f"{name}-P{P}-group{hk}", errs)
        bad = {n: e for n, e in errs.items() if not e <= H.TOL["bf16"]}
        assert not bad, (hk, bad)
