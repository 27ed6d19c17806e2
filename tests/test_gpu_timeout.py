"""The timeout path of the bounded device-side waits, driven on the GPU without a fault or a
hang: gdn_debug_wait_probe launches one CTA whose mbarrier is armed for bytes that no copy
ever delivers (nothing is in flight), so its bounded wait runs out after a short, given number
of polls. The CTA then records GDN_ERR_TIMEOUT in the device status word and frees its tensor
memory, as every kernel of the library does when a wait runs out; the context must stay
usable, and the next calls must be correct."""
import os

import pytest

import gdn_synthetic as gs
import gpu_harness as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TIMEOUT = -6


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    import gated_delta_rule_22_gb300 as g
    return g


def test_wait_runs_out_then_context_is_usable(gdn):
    assert gdn.gdn_device_status() == 0
    gdn.gdn_debug_wait_probe(1000)
    assert gdn.gdn_device_status() == TIMEOUT
    assert gdn.gdn_device_status() == 0                 # read and cleared
    # twice in a row, and each time the tensor memory it held is free again for the kernels
    gdn.gdn_debug_wait_probe(10)
    gdn.gdn_debug_wait_probe(10)
    assert gdn.gdn_device_status() == TIMEOUT
    for w in (gs.Workload("after-tc", 1, 150, 1, 2, 128, 128, "bf16", "strong", True, True, 64),
              gs.Workload("after-seq", 1, 40, 2, 4, 64, 32, "f32", "weak", True, True, 16)):
        inp = gs.make_inputs(w)
        errs = H.errors(H.to_numpy(H.run_gpu(inp)), H.run_oracle(inp))
        assert all(e <= H.TOL[w.dtype] for e in errs.values()), (w.name, errs)
    assert gdn.gdn_device_status() == 0


def test_fma_rate_is_measured(gdn):
    """The FP32 FMA rate that bench.py uses as the sequential kernels' peak: positive and below
    what 152 SMs x 128 lanes x 2 flop could give at 2.2 GHz."""
    for packed in (False, True):
        r = gdn.gdn_diag_fma_tflops(packed)
        assert 10.0 < r < 152 * 128 * 2 * 2.2e9 / 1e12, (packed, r)
