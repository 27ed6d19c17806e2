"""Host checks of bench.py's bookkeeping: the source hash that keys the measured DRAM traffic,
the per-kernel roofline choice, and the gradient kernels' split-group bytes against the
kernels' own cover of the value-head groups (mirrored in test_chunk_split_groups)."""
import os

import pytest

import bench
import gdn_synthetic as gs
from test_chunk_split_groups import ranges, written_parts

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


@pytest.mark.parametrize("name", [n for n, w in gs.WORKLOADS.items() if w.dtype == "bf16"])
def test_split_group_bytes_bound_the_kernels_cover(name):
    """bench.py counts, per CTA boundary, two fp32 [dq; dk] parts (gradient kernel writes,
    reduction reads) and one bf16 group (reduction writes): an upper bound on what the
    kernels' unit ranges actually split, for a GB300's 152 SMs."""
    w = gs.WORKLOADS[name]
    NC = -(-w.T // w.chunk)
    units, rep, L, Dk = w.B * NC * w.Hv, w.Hv // w.Hk, w.chunk, w.Dk
    ctas = min(units, 152)
    assert len(ranges(units, ctas)) == ctas
    parts, _ = written_parts(units, ctas, rep, w.Hv)
    n_groups = len({g for g, _ in parts})
    m = bench.kernel_model(w, sms=152)
    part_bytes = 2 * L * Dk * 4                     # dq and dk partial of one part, fp32
    assert len(parts) * part_bytes <= m["chunk_reduce"][0] - n_groups * 2 * L * Dk * 2
    n_split = min(units, 152) - 1
    assert n_groups <= n_split
    assert m["chunk_reduce"][0] == pytest.approx(n_split * (2 * part_bytes + 2 * L * Dk * 2))
