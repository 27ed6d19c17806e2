"""GPU parity of the chunkwise tensor-core forward (bf16 inputs, checkpoint interval 64, the
supported key / value widths), through the C ABI, against the float64 oracle: ragged last
chunks, GQA, a start state and a final-state cotangent, every supported key width, value
widths of one and three 64-row blocks, and the degenerate decays (g = 0 and beta = 0
exactly). The backward consumes the chunkwise forward's checkpoints and residuals, so the
gradients are checked too. Tolerance 5e-3 relative L2 (bf16 inputs)."""
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
    import os
    from gated_delta_rule_22_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_22_gb300 import build
        build.build()
    return torch.device("cuda:0")


CASES = [
    gs.Workload("tc-Dk64-Dv64-ragged", 2, 130, 2, 4, 64, 64, "bf16", "strong", True, True, 64),
    gs.Workload("tc-Dk128-Dv192-gqa3", 1, 200, 2, 6, 128, 192, "bf16", "weak", True, True, 64),
    gs.Workload("tc-Dk192-Dv64-half", 2, 64, 1, 2, 192, 64, "bf16", "half", False, True, 64),
    gs.Workload("tc-Dk192-short", 1, 5, 1, 2, 192, 128, "bf16", "weak", True, False, 64),
    # three batch rows with a ragged last chunk each and no GQA: the persistent gradient
    # kernel's unit ranges cross batch rows and kv heads
    gs.Workload("tc-B3-ragged-noGQA", 3, 190, 3, 3, 128, 128, "bf16", "strong", True, True, 64),
    # 24 value heads on one kv head: dq, dk of each chunk are the sum of 24 heads, all taken by
    # one gradient CTA
    gs.Workload("tc-gqa24", 1, 100, 1, 24, 64, 64, "bf16", "weak", True, True, 64),
    # the chunked backward does not fit shared memory here: the sequential backward consumes
    # the chunkwise forward's saved buffer
    gs.Workload("tc-fwd-seq-bwd-Dv256", 1, 150, 1, 2, 128, 256, "bf16", "half", True, True, 64),
]


def _check(w, inp, dev):
    got = H.to_numpy(H.run_gpu(inp, dev))
    ref = H.run_oracle(inp)
    errs = H.errors(got, ref)
    print(w.name, {n: f"{e:.2e}" for n, e in errs.items()})
    bad = {n: e for n, e in errs.items() if not e <= H.TOL["bf16"]}
    assert not bad, (w.name, bad)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_chunkwise_forward_parity(dev, w):
    _check(w, gs.make_inputs(w), dev)


def test_chunkwise_forward_degenerate_gates(dev):
    """g = 0 (the state is wiped) and beta = 0 (no write) at chosen steps, exactly."""
    w = gs.Workload("tc-degenerate", 1, 150, 1, 2, 128, 64, "bf16", "weak", True, True, 64)
    inp = gs.make_inputs(w)
    g, beta = inp["g"].copy(), inp["beta"].copy()
    g[0, [0, 17, 63, 64, 100], :] = 0.0
    beta[0, [5, 64, 127, 149], :] = 0.0
    inp["g"], inp["beta"] = g, beta
    _check(w, inp, dev)


def test_chunkwise_forward_is_deterministic(dev):
    w = CASES[1]
    inp = gs.make_inputs(w)
    a = H.run_gpu(inp, dev)
    b = H.run_gpu(inp, dev)
    for n in a:
        if a[n] is not None:
            assert torch.equal(a[n], b[n]), n
