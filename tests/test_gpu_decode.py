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
