"""The chunkwise (dense) form of the recurrence and its VJP (tests/chunkwise_form.py) against
the sequential float64 oracle.

1. In float64 the chunkwise form is the same function: every output (y, S_T, checkpoints and
   all gradients, dg under strong decay included) agrees with the oracle to rounding, on
   ragged multi-chunk shapes with GQA, a start state and a final-state cotangent. This pins
   the derivation a chunked tensor-core kernel would implement, including its division-free
   dg (mlx issue #4614 reports a chunked kernel whose dg under strong decay was off by 1e2).
2. With its matrix-product operands cut to tf32 (mantissa truncated to 10 bits) or rounded
   to bf16, as tensor-core operands would be, on bf16-rounded inputs, every output stays
   within the bf16 parity bound of 5e-3 relative L2 (tf32 at about 1e-3, bf16 at about
   3e-3): the precision plan of a tensor-core version for bf16 inputs.
"""
import numpy as np
import pytest

import chunkwise_form as CF
import gdn_synthetic as gs
import oracle


def _run(w):
    inp = gs.make_inputs(w)
    a = [inp[n].astype(np.float64) for n in ("q", "k", "v", "g", "beta")]
    dy = inp["dy"].astype(np.float64)
    S0 = None if inp["S0"] is None else inp["S0"].astype(np.float64)
    dS = None if inp["dS_T"] is None else inp["dS_T"].astype(np.float64)
    return a, dy, S0, dS


@pytest.mark.parametrize("decay", ["weak", "strong", "half"])
def test_chunkwise_form_is_the_recurrence(decay):
    w = gs.Workload("cw", 2, 37, 2, 4, 16, 12, "f32", decay, True, True, 16)
    a, dy, S0, dS = _run(w)
    fo = oracle.fwd(*a, S0, chunk=16)
    bo = oracle.bwd(*a, dy, S0, dS, chunk=16)
    fc = CF.forward(*a, S0, chunk=16)
    bc = CF.backward(*a, dy, S0, dS, chunk=16)
    errs = {n: oracle.rel_l2(fc[n], fo[n]) for n in ("y", "S_T", "ckpt")}
    errs.update({n: oracle.rel_l2(bc[n], bo[n]) for n in bo})
    assert all(e <= 1e-12 for e in errs.values()), errs


def test_chunkwise_residual_is_v_minus_prediction():
    """The chunk's prediction U reproduces the recurrence's u_t = g_t S_{t-1} k_t: checked by
    rebuilding delta = beta (v - u) and the next state step by step from the checkpoint."""
    w = gs.Workload("cw", 1, 20, 1, 2, 8, 6, "f32", "strong", True, False, 8)
    a, _, S0, _ = _run(w)
    q, k, v, g, beta = a
    fc = CF.forward(q, k, v, g, beta, S0, chunk=8)
    for h in range(2):
        S = S0[0, h].copy()
        for t in range(20):
            u = g[0, t, h] * S @ k[0, t, 0]
            assert np.allclose(fc["resid"][0, t, h], v[0, t, h] - u, rtol=1e-12, atol=1e-13)
            S = g[0, t, h] * S + np.outer(beta[0, t, h] * (v[0, t, h] - u), k[0, t, 0])


def _tf32(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return u.view(np.float32).astype(np.float64)


def _bf16(x):
    return gs.round_to_bf16(np.asarray(x, dtype=np.float32)).astype(np.float64)


@pytest.mark.parametrize("decay", ["weak", "strong"])
@pytest.mark.parametrize("name,rnd,bound", [("tf32", _tf32, 2e-3), ("bf16", _bf16, 4e-3)])
def test_low_precision_operands_meet_the_bf16_bound(decay, name, rnd, bound):
    w = gs.Workload("cw", 1, 256, 2, 8, 64, 32, "bf16", decay, False, False, 64)
    a, dy, _, _ = _run(w)
    fo = oracle.fwd(*a, chunk=64)
    bo = oracle.bwd(*a, dy, chunk=64)
    fc = CF.forward(*a, chunk=64, rnd=rnd)
    bc = CF.backward(*a, dy, chunk=64, rnd=rnd)
    # outputs in the input dtype, as a kernel would write them
    errs = {"y": oracle.rel_l2(_bf16(fc["y"]), fo["y"])}
    errs.update({n: oracle.rel_l2(_bf16(bc[n]) if n != "dS0" else bc[n], bo[n]) for n in bo})
    assert all(e <= 5e-3 for e in errs.values()), (name, decay, errs)
    raw = {n: oracle.rel_l2(bc[n], bo[n]) for n in bo}
    assert all(e <= bound for e in raw.values()), (name, decay, raw)


def test_chunk_state_map_is_the_affine_part():
    """S_L(S0) - S_L(0) = S0 M for the chunk's state map M, on a random start state (a wrong
    sign, decay or transposition in M fails it)."""
    w = gs.Workload("map", 1, 48, 1, 1, 16, 12, "f32", "half", True, False, 48)
    a, _, S0, _ = _run(w)
    q, k, v, g, beta = a
    K, Q, V, gg, bb = k[0, :, 0], q[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0]
    _, SL, _, _, _ = CF.chunk_forward(S0[0, 0], K, Q, V, gg, bb)
    _, SL0, _, _, _ = CF.chunk_forward(np.zeros_like(S0[0, 0]), K, Q, V, gg, bb)
    M = CF.chunk_state_map(K, gg, bb)
    assert np.allclose(SL - SL0, S0[0, 0] @ M, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("segments", [1, 2, 3, 5])
@pytest.mark.parametrize("decay", ["weak", "strong"])
def test_segment_scan_is_the_recurrence(segments, decay):
    """The forward and the VJP as scans over segments of chunks (the sequence-parallel form)
    agree with the sequential oracle to rounding, on a ragged GQA shape with a start state and a
    final-state cotangent."""
    w = gs.Workload("seg", 1, 86, 1, 2, 12, 10, "f32", decay, True, True, 16)
    a, dy, S0, dS = _run(w)
    fo = oracle.fwd(*a, S0, chunk=16)
    bo = oracle.bwd(*a, dy, S0, dS, chunk=16)
    fs = CF.forward_segments(*a, S0, chunk=16, segments=segments)
    bs = CF.backward_segments(*a, dy, S0, dS, chunk=16, segments=segments)
    errs = {n: oracle.rel_l2(fs[n], fo[n]) for n in ("y", "S_T", "ckpt")}
    errs.update({n: oracle.rel_l2(bs[n], bo[n]) for n in bo})
    assert all(e <= 1e-11 for e in errs.values()), errs
