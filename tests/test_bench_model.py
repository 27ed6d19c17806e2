"""Host checks of bench.py's bookkeeping: the source hash that keys the measured DRAM traffic,
the per-kernel roofline choice, and the per-kernel algorithmic bytes (each tensor of the
method's byte count attributed to exactly one kernel of its pass)."""
import os

import pytest

import bench
import gdn_synthetic as gs

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "gated_delta_rule_22_gb300", "csrc")


def test_kernel_files_exist():
    for name, files in bench.KERNEL_FILES.items():
        for f in files:
            assert os.path.isfile(os.path.join(CSRC, f)), (name, f)


def test_code_hash_ignores_comments_and_layout_only():
    src = open(os.path.join(CSRC, "gdn_chunk_bwd.cu"), encoding="utf-8").read()
    commented = ("/* a block comment\n   over two lines */\n" + src.replace("\n", "   // note\n", 3)
                 .replace("namespace gdn {", "namespace   gdn\n\n{", 1))
    assert bench._code_only(commented) == bench._code_only(src)
    edited = src.replace("kL = 64;", "kL = 32;", 1)
    assert edited != src and bench._code_only(edited) != bench._code_only(src)


def test_traffic_lookup_is_keyed_by_the_family_sources():
    for name in bench.KERNEL_FILES:
        got = bench.traffic_of(name)
        assert got is None or got > 0
    assert bench.traffic_of("no_such_kernel") is None


def test_roofline_takes_the_slowest_bound():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    # 1 GB at 1000 GB/s = 1 ms; 50 TFLOP at 100 TFLOP/s = 500 ms: tensor-bound
    r = bench.kernel_roofline("k", 1000.0, (1e9, 50e12, 0.0), peaks)
    assert r["bound"] == "tensor" and r["roofline_ms"] == pytest.approx(500.0)
    assert r["achieved"] == pytest.approx(50.0) and r["frac"] == pytest.approx(0.5)
    r = bench.kernel_roofline("k", 2.0, (1e9, 1e9, 0.0), peaks)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(500.0) and r["frac"] == pytest.approx(0.5)


FWD = {"q", "k", "v", "g", "beta", "S0", "y", "S_T", "ckpt"}
BWD = {"q", "k", "v", "g", "beta", "ckpt", "dy", "dS_T", "dq", "dk", "dv", "dg", "dbeta", "dS0"}


@pytest.mark.parametrize("kernels,tensors", [
    (("chunk_prep", "chunk_sweep"), FWD), (("chunk_dsweep", "chunk_grad"), BWD),
    (("seq_fwd",), FWD), (("seq_bwd", "seq_reduce"), BWD),
])
def test_each_tensor_of_a_pass_credited_to_one_kernel(kernels, tensors):
    got = [n for k in kernels for n in bench.PASS_TENSORS[k]]
    assert sorted(got) == sorted(tensors)


@pytest.mark.parametrize("name", sorted(gs.WORKLOADS))
def test_kernel_bytes_add_up_to_the_step(name):
    w = gs.WORKLOADS[name]
    m = bench.kernel_model(w)
    step = bench.bytes_per_step(w)
    assert sum(m[k][0] for k in ("chunk_prep", "chunk_sweep", "chunk_dsweep", "chunk_grad")) == pytest.approx(step)
    assert sum(m[k][0] for k in ("seq_fwd", "seq_bwd", "seq_reduce")) == pytest.approx(step)


def test_step_bytes_at_the_headline_shape():
    """linattn-T2048 (no S0, no dS_T): q, k 12.6 MB each, v, y, dy, dv 33.6 MB each, checkpoints
    32 x 6.29 MB: 660.1 MB per step."""
    w = gs.WORKLOADS["linattn-T2048"]
    assert bench.bytes_per_step(w) == pytest.approx(660.1e6, rel=1e-3)
