"""Inference and decode forward: gdn_fwd without a saved-for-backward buffer (ckpt = NULL).

A forward without checkpoints is the same forward (bitwise), and a decode loop of T = 1
steps, each passing the carried state as S0 and reading it back from S_T, reproduces the
float64 oracle's forward over the whole sequence (the recurrence of mlx issue #4614,
"Recurrence used for the references", applied one step at a time)."""
import pytest

import gdn_synthetic as gs
import gpu_harness as H
import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return torch.device("cuda:0")


def test_forward_without_checkpoints_is_the_same_forward(dev):
    import gated_delta_rule_22_gb300 as gdn
    w = gs.Workload("nockpt", 2, 77, 2, 6, 96, 24, "f32", "strong", True, False, 16)
    t = H.to_device(gs.make_inputs(w), dev)
    y0, S0_T, ck = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], chunk=16)
    y1, S1_T, none = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], chunk=16,
                                 want_ckpt=False)
    torch.cuda.synchronize()
    assert none is None and ck is not None
    assert torch.equal(y0, y1) and torch.equal(S0_T, S1_T)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_match_the_oracle(dev, dtype):
    import gated_delta_rule_22_gb300 as gdn
    w = gs.Workload("decode", 2, 24, 2, 4, 64, 32, dtype, "weak", True, False)
    inp = gs.make_inputs(w)
    t = H.to_device(inp, dev)
    S = t["S0"]
    ys = []
    for step in range(w.T):
        cut = {n: t[n][:, step:step + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        y, S, ck = gdn.gdn_fwd(cut["q"], cut["k"], cut["v"], cut["g"], cut["beta"], S, want_ckpt=False)
        assert ck is None
        ys.append(y)
    y = torch.cat(ys, dim=1)
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk)
    tol = H.TOL[dtype]
    e_y = oracle.rel_l2(y.double().cpu().numpy(), ref["y"])
    e_s = oracle.rel_l2(S.double().cpu().numpy(), ref["S_T"])
    assert e_y <= tol and e_s <= tol, (dtype, e_y, e_s)


@pytest.mark.parametrize("name", ["decode-B1", "decode-B64"])
def test_decode_step_at_the_benchmark_shapes(dev, name):
    """One decode step of the layer (Hv = 64 on Hk = 16, Dk = 192, Dv = 128) for 1 and 64
    sequences, as `bench.py --workload decode-B*` times it: y and the carried state, whole
    tensors, against the oracle."""
    import gated_delta_rule_22_gb300 as gdn
    w = gs.WORKLOADS[name]
    inp = gs.make_inputs(w)
    t = H.to_device(inp, dev)
    y, S_T, ck = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], want_ckpt=False)
    torch.cuda.synchronize()
    assert ck is None
    ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk)
    e_y = oracle.rel_l2(y.double().cpu().numpy(), ref["y"])
    e_s = oracle.rel_l2(S_T.double().cpu().numpy(), ref["S_T"])
    print(name, f"y {e_y:.2e} S_T {e_s:.2e}")
    assert e_y <= H.TOL["bf16"] and e_s <= H.TOL["bf16"], (e_y, e_s)


@pytest.mark.parametrize("w", [
    gs.Workload("dec-f32-Dv40-noS0", 3, 1, 2, 6, 128, 40, "f32", "strong", False, False),
    gs.Workload("dec-f32-Dk256", 2, 1, 1, 2, 256, 64, "f32", "weak", True, False),
    gs.Workload("dec-bf16-Dk96-seq", 2, 1, 1, 3, 96, 64, "bf16", "weak", True, False),   # the sequential kernel
    gs.Workload("dec-bf16-gqa8", 1, 1, 1, 8, 64, 200, "bf16", "half", True, False),
], ids=lambda w: w.name)
def test_decode_step_shapes(dev, w):
    """The decode step on ragged value widths, no incoming state, every key width it takes (and
    one it leaves to the sequential kernel), GQA; the state updated in place gives the same."""
    import gated_delta_rule_22_gb300 as gdn
    inp = gs.make_inputs(w)
    t = H.to_device(inp, dev)
    y, S_T, _ = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], want_ckpt=False)
    ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk)
    tol = H.TOL[w.dtype]
    e_y = oracle.rel_l2(y.double().cpu().numpy(), ref["y"])
    e_s = oracle.rel_l2(S_T.double().cpu().numpy(), ref["S_T"])
    assert e_y <= tol and e_s <= tol, (e_y, e_s)
    if t["S0"] is not None:
        S = t["S0"].clone()
        y2, S2, _ = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], S, S_T=S, want_ckpt=False)
        torch.cuda.synchronize()
        assert torch.equal(y2, y) and torch.equal(S, S_T)


@pytest.mark.parametrize("w", [
    gs.Workload("inf-Dk64-Dv64-ragged", 2, 130, 2, 4, 64, 64, "bf16", "strong", True, False),
    gs.Workload("inf-Dk128-Dv256", 1, 200, 1, 2, 128, 256, "bf16", "weak", True, False),
    gs.Workload("inf-Dk192-gqa", 1, 300, 2, 6, 192, 128, "bf16", "half", False, False),
    gs.WORKLOADS["linattn-T2048"],
], ids=lambda w: w.name)
def test_inference_forward_is_the_forward(dev, w):
    """gdn_fwd_infer (the chunkwise forward with nothing saved) gives y and S_T bit for bit as
    gdn_fwd does with its saved buffer, and matches the oracle."""
    import gated_delta_rule_22_gb300 as gdn
    inp = gs.make_inputs(w)
    t = H.to_device(inp, dev)
    y, S_T = gdn.gdn_fwd_infer(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"])
    y0, S0_T, _ = gdn.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"])
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(S_T, S0_T)
    if w.T <= 300:
        ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"], chunk=w.chunk)
        e_y = oracle.rel_l2(y.double().cpu().numpy(), ref["y"])
        e_s = oracle.rel_l2(S_T.double().cpu().numpy(), ref["S_T"])
        assert e_y <= H.TOL["bf16"] and e_s <= H.TOL["bf16"], (e_y, e_s)
