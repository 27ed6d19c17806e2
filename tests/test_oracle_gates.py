"""Pins of the oracle's gate functions (oracle.gates_fwd / oracle.gates_bwd), none of which
uses the oracle's own arithmetic for the expected value:

* central finite differences of the gate map in float64, element by element for a and b
  and per head for A_log and dt_bias;
* closed forms: softplus(0) = log 2 (g = 2^-exp(A_log)), sigmoid(0) = 1/2, the saturated
  ends (a + dt_bias -> -inf or A_log -> -inf give g = 1; large a + dt_bias gives
  g = exp(-exp(A_log) (a + dt_bias)));
* the sum rule ddt_bias[h] = sum over rows of da[., h] (dt_bias enters only through
  a + dt_bias);
* finite differences of the whole chain: gate map -> recurrence -> <dy, y>, with the
  recurrence's dg and dbeta fed into gates_bwd (the eight trainable inputs of mlx-lm PR
  #1217, "Correctness": q, k, v, a, b, A_log, dt_bias and the state);
* planted mistakes in copies of the oracle source, each caught by the pins above.
"""
import numpy as np
import pytest

import gdn_synthetic as gs
import oracle


def _inputs(decay="weak", B=2, T=7, Hv=5, seed=3):
    w = gs.Workload("gates", B, T, 1, Hv, 32, 32, "f32", decay, seed=seed)
    gi = gs.make_gate_inputs(w)
    return {n: gi[n].astype(np.float64) for n in ("a", "b", "A_log", "dt_bias", "dg", "dbeta")}


def _fd_gates(x, lib=None, h=1e-6):
    """Central differences of L = <dg, g> + <dbeta, beta> (dg, dbeta as fixed weights)."""
    def L(a, b, A_log, dt_bias):
        f = oracle.gates_fwd(a, b, A_log, dt_bias, lib=lib)
        return f["g"], f["beta"]

    a, b, A_log, dt_bias = x["a"], x["b"], x["A_log"], x["dt_bias"]
    gp, _ = L(a + h, b, A_log, dt_bias)
    gm, _ = L(a - h, b, A_log, dt_bias)
    da = x["dg"] * (gp - gm) / (2 * h)          # g[i] depends on a[i] only
    _, bp = L(a, b + h, A_log, dt_bias)
    _, bm = L(a, b - h, A_log, dt_bias)
    db = x["dbeta"] * (bp - bm) / (2 * h)
    dA = np.empty_like(A_log)
    dd = np.empty_like(dt_bias)
    for hh in range(A_log.size):
        e = np.zeros_like(A_log)
        e[hh] = h
        dA[hh] = np.sum(x["dg"] * (L(a, b, A_log + e, dt_bias)[0] - L(a, b, A_log - e, dt_bias)[0])) / (2 * h)
        dd[hh] = np.sum(x["dg"] * (L(a, b, A_log, dt_bias + e)[0] - L(a, b, A_log, dt_bias - e)[0])) / (2 * h)
    return {"da": da, "db": db, "dA_log": dA, "ddt_bias": dd}


def pin_gates_fd(lib=None, tol=1e-7):
    for decay in ("weak", "strong"):
        x = _inputs(decay)
        got = oracle.gates_bwd(x["a"], x["b"], x["A_log"], x["dt_bias"], x["dg"], x["dbeta"], lib=lib)
        want = _fd_gates(x, lib)
        for n in want:
            e = oracle.rel_l2(got[n], want[n])
            if not e <= tol:
                return f"{decay} {n}: rel L2 {e:.3g} vs finite differences"
    return None


def pin_gates_closed_forms(lib=None):
    Hv = 4
    A_log = np.array([0.0, 0.3, -0.7, 1.1])
    dt_bias = np.array([0.25, -0.5, 0.0, 1.5])
    # a + dt_bias = 0: softplus = log 2, so g = 2^-exp(A_log); b = 0: beta = 1/2
    a = np.tile(-dt_bias, (3, 1))
    f = oracle.gates_fwd(a, np.zeros_like(a), A_log, dt_bias, lib=lib)
    if not np.allclose(f["g"], np.tile(2.0 ** -np.exp(A_log), (3, 1)), rtol=1e-14, atol=0):
        return "g at a + dt_bias = 0 is not 2^-exp(A_log)"
    if not np.all(f["beta"] == 0.5):
        return "beta at b = 0 is not 1/2"
    ones = np.ones_like(a)
    d = oracle.gates_bwd(a, np.zeros_like(a), A_log, dt_bias, ones, ones, lib=lib)
    if not np.allclose(d["db"], 0.25, rtol=1e-15, atol=0):
        return "dbeta/db at b = 0 is not 1/4"
    # d(log g)/da = -exp(A_log) * sigmoid(0) = -exp(A_log)/2, times g
    want_da = np.tile(2.0 ** -np.exp(A_log) * -np.exp(A_log) / 2, (3, 1))
    if not np.allclose(d["da"], want_da, rtol=1e-14, atol=0):
        return "da at a + dt_bias = 0 is not -g exp(A_log)/2"
    # saturated ends
    far = oracle.gates_fwd(np.full((2, Hv), -80.0), np.zeros((2, Hv)), A_log, np.zeros(Hv), lib=lib)
    if not np.all(far["g"] == 1.0):
        return "g is not 1 for a + dt_bias -> -inf"
    tiny = oracle.gates_fwd(np.full((2, Hv), 3.0), np.zeros((2, Hv)), np.full(Hv, -80.0), np.zeros(Hv), lib=lib)
    if not np.all(tiny["g"] == 1.0):
        return "g is not 1 for A_log -> -inf"
    big = oracle.gates_fwd(np.full((2, Hv), 45.0), np.zeros((2, Hv)), A_log, np.zeros(Hv), lib=lib)
    if not np.allclose(big["g"], np.tile(np.exp(-np.exp(A_log) * 45.0), (2, 1)), rtol=1e-12, atol=0):
        return "g is not exp(-exp(A_log) x) for large x"
    return None


def pin_gates_sum_rule(lib=None):
    x = _inputs("strong")
    d = oracle.gates_bwd(x["a"], x["b"], x["A_log"], x["dt_bias"], x["dg"], x["dbeta"], lib=lib)
    want = d["da"].reshape(-1, d["da"].shape[-1]).sum(axis=0)
    if not np.allclose(d["ddt_bias"], want, rtol=1e-12, atol=1e-300):
        return "ddt_bias is not the row sum of da"
    return None


GATE_PINS = [pin_gates_closed_forms, pin_gates_sum_rule, pin_gates_fd]


@pytest.mark.parametrize("pin", GATE_PINS, ids=lambda p: p.__name__)
def test_gate_pin(pin):
    assert pin() is None


@pytest.mark.parametrize("decay", ["weak", "strong"])
def test_chain_through_the_recurrence(decay):
    """FD of <dy, y> with g, beta from the gate map, against gates_bwd fed with the
    recurrence's own dg and dbeta."""
    rng = np.random.default_rng(11)
    w = gs.Workload("chain", 1, 9, 1, 2, 8, 6, "f32", decay, seed=5)
    inp = gs.make_inputs(w)
    x = _inputs(decay, B=1, T=9, Hv=2, seed=5)
    q, k, v, dy = (inp[n].astype(np.float64) for n in ("q", "k", "v", "dy"))

    def L(a, b, A_log, dt_bias):
        f = oracle.gates_fwd(a, b, A_log, dt_bias)
        return oracle.loss(oracle.fwd(q, k, v, f["g"], f["beta"], chunk=4), dy)

    f = oracle.gates_fwd(x["a"], x["b"], x["A_log"], x["dt_bias"])
    r = oracle.bwd(q, k, v, f["g"], f["beta"], dy, chunk=4)
    d = oracle.gates_bwd(x["a"], x["b"], x["A_log"], x["dt_bias"], r["dg"], r["dbeta"])
    h = 1e-6
    args = {n: x[n].copy() for n in ("a", "b", "A_log", "dt_bias")}
    for name, grad in (("a", "da"), ("b", "db"), ("A_log", "dA_log"), ("dt_bias", "ddt_bias")):
        flat = args[name].reshape(-1)
        idx = range(flat.size) if flat.size <= 4 else rng.choice(flat.size, 6, replace=False)
        for i in idx:
            old = flat[i]
            flat[i] = old + h
            lp = L(**args)
            flat[i] = old - h
            lm = L(**args)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            got = d[grad].reshape(-1)[i]
            assert abs(got - fd) <= 1e-6 * max(1.0, abs(fd)), (decay, name, i, got, fd)


MUTANTS = [
    ("sigmoid of -x", "dlog_g * (-A) * sigmoid_d(x);", "dlog_g * (-A) * sigmoid_d(-x);", 1),
    ("dA_log misses log g", "dA_log[h] += dlog_g * log_g;", "dA_log[h] += dlog_g;", 1),
    ("d(log g) divides by g", "exp(log_g) * dg[o];", "dg[o] / exp(log_g);", 1),
    ("sigmoid derivative", "db[o] = dbeta[o] * bt * (1.0 - bt);", "db[o] = dbeta[o] * bt;", 1),
    ("dt_bias not accumulated", "ddt_bias[h] += dx;", "ddt_bias[h] = dx;", 1),
    ("forward subtracts dt_bias", "softplus_d(a[o] + dt_bias[h]);", "softplus_d(a[o] - dt_bias[h]);", 1),
    ("forward drops exp of A_log", "const double log_g = -exp(A_log[h]) * softplus_d",
     "const double log_g = -A_log[h] * softplus_d", 1),
]


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_gate_mutant_is_caught(tmp_path, name, old, new, count):
    source = open(oracle._SRC).read()
    assert source.count(old) == count, f"mutation '{name}' no longer matches the oracle source"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.build(str(src), so)
    lib = oracle.load(so)
    for pin in GATE_PINS:
        if pin(lib) is not None:
            return
    pytest.fail(f"mutant '{name}' passed every gate pin")
