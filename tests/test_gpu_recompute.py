"""GPU parity of the re-computation mode (gdn_fwd_rc / gdn_bwd_rc): the saved buffer holds only
the fp32 chunk-start states and the residuals, and the backward forms the chunkwise products
again. Every output -- y, S_T, the checkpoints and all gradients -- equals that of gdn_fwd /
gdn_bwd bit for bit (the same kernels on the same inputs; the checkpoints' bf16 operand copies
round the same fp32 values the forward sweep rounds), on ragged and GQA shapes, every key width,
value widths of one to three 64-row blocks, at the headline shape at full size, and against the
float64 oracle within the bf16 bound."""
import os

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


def run_rc(inp, dev):
    import gated_delta_rule_22_gb300 as gdn
    t = H.to_device(inp, dev)
    y, S_T, ck = gdn.gdn_fwd_rc(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"])
    gr = gdn.gdn_bwd_rc(t["q"], t["k"], t["v"], t["g"], t["beta"], ck, t["dy"], t["dS_T"])
    torch.cuda.synchronize()
    return {"y": y, "S_T": S_T, "ckpt": ck, **gr}


CASES = [
    gs.Workload("rc-Dk64-Dv64-ragged", 2, 130, 2, 4, 64, 64, "bf16", "strong", True, True, 64),
    gs.Workload("rc-Dk128-Dv192-gqa3", 1, 200, 2, 6, 128, 192, "bf16", "weak", True, True, 64),
    gs.Workload("rc-Dk192-Dv64-half", 2, 64, 1, 2, 192, 64, "bf16", "half", False, True, 64),
    gs.Workload("rc-B3-ragged-noGQA", 3, 190, 3, 3, 128, 128, "bf16", "strong", True, True, 64),
    gs.WORKLOADS["linattn-T2048"],
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_recompute_mode_equals_the_saved_products_mode(dev, w):
    inp = gs.make_inputs(w)
    a = run_rc(inp, dev)
    b = H.run_gpu(inp, dev)
    for n in H.OUTPUTS:
        if b.get(n) is None:
            continue
        assert torch.equal(a[n], b[n]), n


def test_recompute_mode_against_the_oracle(dev):
    w = gs.Workload("rc-oracle", 1, 300, 2, 4, 192, 128, "bf16", "strong", True, True, 64)
    inp = gs.make_inputs(w)
    got = H.to_numpy(run_rc(inp, dev))
    errs = H.errors(got, H.run_oracle(inp))
    print(errs)
    assert set(errs) == set(H.OUTPUTS), errs
    bad = {n: e for n, e in errs.items() if not e <= H.TOL["bf16"]}
    assert not bad, bad


def test_recompute_saved_buffer_is_smaller(dev):
    import gated_delta_rule_22_gb300 as gdn
    w = gs.WORKLOADS["linattn-T2048"]
    s = gdn.make_shape(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, 64, gdn.GDN_BF16)
    states = w.B * w.Hv * (w.T // 64) * w.Dv * w.Dk * 4
    resid = w.B * w.T * w.Hv * w.Dv * 4
    assert gdn.gdn_rc_ckpt_bytes(s) == states + resid
    assert gdn.gdn_rc_ckpt_bytes(s) < 0.55 * gdn.gdn_ckpt_bytes(s)
