"""The library's per-kernel timing (gdn_timing_enable / gdn_timing_read): it records each
kernel family the calls launch, with positive device times, nothing while it is off, and
it clears the record on every read."""
import pytest

import gdn_synthetic as gs
import gpu_harness as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    import gated_delta_rule_22_gb300 as g
    return g


def _step(g, w):
    t = H.to_device(gs.make_inputs(w), torch.device("cuda:0"))
    _, _, ckpt = g.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"], chunk=w.chunk)
    g.gdn_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], ckpt, t["dy"], t["dS_T"], chunk=w.chunk)
    torch.cuda.synchronize()


@pytest.mark.parametrize("w,names", [
    (gs.Workload("tc", 1, 130, 1, 2, 128, 128, "bf16", "weak", True, True, 64),
     ["chunk_prep", "chunk_sweep", "chunk_dsweep", "chunk_grad"]),
    (gs.Workload("seq", 1, 40, 1, 2, 64, 32, "f32", "weak", False, False, 16),
     ["seq_fwd", "seq_bwd", "seq_reduce"]),
])
def test_timing_records_each_kernel(gdn, w, names):
    gdn.gdn_timing_read()
    gdn.gdn_timing_enable(True)
    try:
        _step(gdn, w)
        _step(gdn, w)
        rec = gdn.gdn_timing_read()
    finally:
        gdn.gdn_timing_enable(False)
    assert list(rec) == names
    for n in names:
        launches, ms = rec[n]
        assert launches == 2 and ms > 0.0, (n, rec[n])
    assert gdn.gdn_timing_read() == {}          # the read cleared the record


def test_timing_off_records_nothing(gdn):
    gdn.gdn_timing_enable(False)
    _step(gdn, gs.Workload("seq", 1, 20, 1, 1, 32, 8, "f32", "weak", False, False, 8))
    assert gdn.gdn_timing_read() == {}
