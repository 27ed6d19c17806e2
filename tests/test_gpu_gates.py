"""GPU parity of the gate map and its VJP (gdn_gates_fwd / gdn_gates_bwd, through the C ABI)
against the float64 oracle, and of the whole chain gates -> recurrence -> gates VJP.

Tolerances as for the recurrence: relative L2 per output <= 1e-5 for float32 inputs and
<= 5e-3 for bf16 inputs (against the oracle run on the bf16-rounded values)."""
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


def _to(gi, dev):
    w = gi["workload"]
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    t = {n: torch.from_numpy(gi[n]).to(dev).to(dt) for n in ("a", "b", "dg", "dbeta")}
    t.update({n: torch.from_numpy(gi[n]).to(dev) for n in ("A_log", "dt_bias")})
    return t


GATE_CASES = [
    gs.Workload("gates-f32-strong", 2, 61, 2, 6, 32, 8, "f32", "strong"),
    gs.Workload("gates-f32-weak", 1, 130, 3, 45, 32, 8, "f32", "weak"),
    gs.Workload("gates-f32-half", 3, 17, 1, 40, 32, 8, "f32", "half"),
    gs.Workload("gates-bf16-batched", 8, 4096, 16, 32, 128, 128, "bf16", "half"),
]


@pytest.mark.parametrize("w", GATE_CASES, ids=lambda w: w.name)
def test_gates_match_the_oracle(dev, w):
    import gated_delta_rule_22_gb300 as gdn
    gi = gs.make_gate_inputs(w)
    t = _to(gi, dev)
    g, beta = gdn.gdn_gates_fwd(t["a"], t["b"], t["A_log"], t["dt_bias"])
    d = gdn.gdn_gates_bwd(t["a"], t["b"], t["A_log"], t["dt_bias"], t["dg"], t["dbeta"])
    torch.cuda.synchronize()
    ref = {**oracle.gates_fwd(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"]),
           **oracle.gates_bwd(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"], gi["dg"], gi["dbeta"])}
    got = {"g": g, "beta": beta, **d}
    tol = H.TOL[w.dtype]
    errs = {n: oracle.rel_l2(got[n].double().cpu().numpy(), ref[n]) for n in ref}
    assert all(e <= tol for e in errs.values()), (w.name, errs)


def test_gates_deterministic(dev):
    import gated_delta_rule_22_gb300 as gdn
    gi = gs.make_gate_inputs(GATE_CASES[-1])
    t = _to(gi, dev)
    runs = [gdn.gdn_gates_bwd(t["a"], t["b"], t["A_log"], t["dt_bias"], t["dg"], t["dbeta"]) for _ in range(2)]
    torch.cuda.synchronize()
    for n in runs[0]:
        assert torch.equal(runs[0][n], runs[1][n]), n


@pytest.mark.parametrize("decay", ["strong", "weak"])
def test_whole_chain_matches_the_oracle(dev, decay):
    """gates -> forward -> backward -> gates VJP on the GPU against the same chain in the
    oracle: gradients for all eight trainable inputs (q, k, v, a, b, A_log, dt_bias, S0)."""
    import gated_delta_rule_22_gb300 as gdn
    w = gs.Workload("chain", 2, 45, 2, 4, 64, 24, "f32", decay, True, False, 16)
    inp = gs.make_inputs(w)
    gi = gs.make_gate_inputs(w)
    t = H.to_device(inp, dev)
    tg = _to(gi, dev)
    g, beta = gdn.gdn_gates_fwd(tg["a"], tg["b"], tg["A_log"], tg["dt_bias"], Hk=w.Hk, Dk=w.Dk, Dv=w.Dv)
    y, S_T, ck = gdn.gdn_fwd(t["q"], t["k"], t["v"], g, beta, t["S0"], chunk=w.chunk)
    r = gdn.gdn_bwd(t["q"], t["k"], t["v"], g, beta, ck, t["dy"], None, chunk=w.chunk)
    d = gdn.gdn_gates_bwd(tg["a"], tg["b"], tg["A_log"], tg["dt_bias"], r["dg"], r["dbeta"],
                          Hk=w.Hk, Dk=w.Dk, Dv=w.Dv)
    torch.cuda.synchronize()
    f = oracle.gates_fwd(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"])
    ro = oracle.bwd(inp["q"], inp["k"], inp["v"], f["g"], f["beta"], inp["dy"], inp["S0"], None, chunk=w.chunk)
    do = oracle.gates_bwd(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"], ro["dg"], ro["dbeta"])
    got = {"dq": r["dq"], "dk": r["dk"], "dv": r["dv"], "dS0": r["dS0"], **d}
    ref = {"dq": ro["dq"], "dk": ro["dk"], "dv": ro["dv"], "dS0": ro["dS0"], **do}
    errs = {n: oracle.rel_l2(got[n].double().cpu().numpy(), ref[n]) for n in ref}
    assert all(e <= H.TOL["f32"] for e in errs.values()), (decay, errs)
