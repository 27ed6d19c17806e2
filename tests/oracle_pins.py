"""Independent checks that pin the float64 oracle to the mathematics of the method.

None of these re-uses the oracle's arithmetic. Each takes an oracle library handle
(`oracle.load(path)`), so the same battery can be pointed at deliberately broken
copies of the oracle (tests/test_oracle_mutants.py) to show that a plausible mistake
in it fails at least one check.

Sources of truth used here:
  * central finite differences of the oracle's own forward (the backward is then
    pinned to the forward), as in the finite-difference test of mlx-lm PR #1217
    "Add Metal VJP kernel for gated_delta_update" (section "Correctness": B=1, T=4,
    Hk=2, Hv=4, Dk=Dv=8) but in float64 and with a much tighter tolerance;
  * forward-mode tangent propagation written out below (a different derivation from
    the reverse sweep), used as a brute-force Jacobian on the toy shape;
  * closed forms of special cases of the recurrence stated on mlx issue #4614
    ("Recurrence used for the references"): g = 0, g = 1 with beta = 0, T = 1,
    orthonormal keys (gated causal linear attention as matrix products), one fixed
    unit key (a first-order linear filter, solved by scipy.signal.lfilter), and
    exact retrieval (beta = 1, unit keys, q = k gives y = v).
"""
from __future__ import annotations

import numpy as np

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def rand_problem(seed, B=1, T=4, Hk=2, Hv=4, Dk=8, Dv=8, S0=True, dST=True, g_range=(0.3, 0.99)):
    """Generic well-conditioned float64 inputs (not the benchmark recipe)."""
    r = _rng(seed)
    p = {
        "q": r.standard_normal((B, T, Hk, Dk)) / np.sqrt(Dk),
        "k": r.standard_normal((B, T, Hk, Dk)) / np.sqrt(Dk),
        "v": r.standard_normal((B, T, Hv, Dv)),
        "g": r.uniform(*g_range, (B, T, Hv)),
        "beta": r.uniform(0.1, 0.9, (B, T, Hv)),
        "dy": r.standard_normal((B, T, Hv, Dv)),
        "S0": r.standard_normal((B, Hv, Dv, Dk)) * 0.3 if S0 else None,
        "dS_T": r.standard_normal((B, Hv, Dv, Dk)) if dST else None,
    }
    return p


def run_fwd(lib, p, chunk=3):
    return oracle.fwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["S0"], chunk=chunk, lib=lib)


def run_bwd(lib, p, chunk=3):
    return oracle.bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["dy"], p["S0"], p["dS_T"],
                      chunk=chunk, lib=lib)


def objective(lib, p, chunk=3):
    return oracle.loss(run_fwd(lib, p, chunk), p["dy"], p["dS_T"])


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "S0": "dS0"}


# --------------------------------------------------------------------------- FD
def pin_finite_differences(lib, p=None, h=1e-6, tol=1e-7, chunk=3):
    """Every element of every input gradient vs a central difference of the forward."""
    if p is None:
        p = rand_problem(1)
    grads = run_bwd(lib, p, chunk)
    worst = 0.0
    for name, gname in GRAD_OF.items():
        if p[name] is None:
            continue
        base = p[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            orig = base[idx]
            base[idx] = orig + h
            lp = objective(lib, p, chunk)
            base[idx] = orig - h
            lm = objective(lib, p, chunk)
            base[idx] = orig
            fd[idx] = (lp - lm) / (2 * h)
        err = oracle.rel_l2(grads[gname], fd)
        worst = max(worst, err)
        if not err < tol:
            return False, f"{gname}: rel L2 vs central differences {err:.3e} >= {tol:.1e}"
    return True, f"worst rel L2 {worst:.2e}"


def pin_directional_fd(lib, seed=2, ndir=3, h=1e-6, tol=1e-7, **shape):
    """Random-direction central differences on a larger, multi-chunk, ragged shape."""
    shape = {"B": 2, "T": 11, "Hk": 2, "Hv": 6, "Dk": 8, "Dv": 12, **shape}
    p = rand_problem(seed, **shape)
    grads = run_bwd(lib, p, chunk=4)
    r = _rng(seed + 100)
    for _ in range(ndir):
        d = {n: (r.standard_normal(p[n].shape) if p[n] is not None else None) for n in GRAD_OF}
        an = sum(float(np.sum(grads[GRAD_OF[n]] * d[n])) for n in GRAD_OF if d[n] is not None)
        pp = {**p, **{n: p[n] + h * d[n] for n in GRAD_OF if d[n] is not None}}
        pm = {**p, **{n: p[n] - h * d[n] for n in GRAD_OF if d[n] is not None}}
        fd = (objective(lib, pp, 4) - objective(lib, pm, 4)) / (2 * h)
        err = abs(an - fd) / max(abs(fd), 1e-300)
        if not err < tol:
            return False, f"directional derivative {an!r} vs FD {fd!r} (rel {err:.2e})"
    return True, "ok"


# --------------------------------------------------------------- forward mode
def tangent_forward(p, t_):
    """Forward-mode derivative of (y, S_T) along the input tangent t_ (dict of arrays or
    None), propagated step by step through the recurrence (product rule on each line)."""
    q, k, v, g, beta = p["q"], p["k"], p["v"], p["g"], p["beta"]
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    rep = Hv // Hk
    z = {n: (t_.get(n) if t_.get(n) is not None else np.zeros_like(p[n]) if p[n] is not None
             else np.zeros((B, Hv, Dv, Dk))) for n in GRAD_OF}
    qh, kh = np.repeat(q, rep, axis=2), np.repeat(k, rep, axis=2)
    qdh, kdh = np.repeat(z["q"], rep, axis=2), np.repeat(z["k"], rep, axis=2)
    S = p["S0"].copy() if p["S0"] is not None else np.zeros((B, Hv, Dv, Dk))
    Sd = z["S0"].copy()
    yd = np.zeros((B, T, Hv, Dv))
    for t in range(T):
        gt, gd = g[:, t, :, None, None], z["g"][:, t, :, None, None]
        A, Ad = gt * S, gd * S + gt * Sd
        kt, kd = kh[:, t, :, None, :], kdh[:, t, :, None, :]
        u = (A * kt).sum(-1)
        ud = (Ad * kt).sum(-1) + (A * kd).sum(-1)
        bt, bd = beta[:, t, :, None], z["beta"][:, t, :, None]
        r_, rd = v[:, t] - u, z["v"][:, t] - ud
        dl, dld = bt * r_, bd * r_ + bt * rd
        S = A + dl[..., None] * kt
        Sd = Ad + dld[..., None] * kt + dl[..., None] * kd
        qt, qd = qh[:, t, :, None, :], qdh[:, t, :, None, :]
        yd[:, t] = (Sd * qt).sum(-1) + (S * qd).sum(-1)
    return yd, Sd


def pin_forward_mode_jacobian(lib, p=None, tol=1e-11, chunk=3):
    """Brute force: each gradient element is the forward-mode derivative of
    <dy, y> + <dS_T, S_T> along that element's basis direction."""
    if p is None:
        p = rand_problem(3)
    grads = run_bwd(lib, p, chunk)
    for name, gname in GRAD_OF.items():
        if p[name] is None:
            continue
        jac = np.empty_like(p[name])
        for idx in np.ndindex(p[name].shape):
            e = np.zeros_like(p[name])
            e[idx] = 1.0
            yd, Sd = tangent_forward(p, {name: e})
            val = float(np.sum(p["dy"] * yd))
            if p["dS_T"] is not None:
                val += float(np.sum(p["dS_T"] * Sd))
            jac[idx] = val
        err = oracle.rel_l2(grads[gname], jac)
        if not err < tol:
            return False, f"{gname}: rel L2 vs forward-mode brute force {err:.3e}"
    return True, "ok"


def pin_dot_product(lib, seed=4, tol=1e-11, **shape):
    """<VJP(dy, dS_T), d> == <(dy, dS_T), JVP(d)> for random d, one input at a time."""
    shape = {"B": 2, "T": 13, "Hk": 3, "Hv": 6, "Dk": 16, "Dv": 8, **shape}
    p = rand_problem(seed, **shape)
    grads = run_bwd(lib, p, chunk=5)
    r = _rng(seed + 7)
    for name, gname in GRAD_OF.items():
        if p[name] is None:
            continue
        d = r.standard_normal(p[name].shape)
        yd, Sd = tangent_forward(p, {name: d})
        rhs = float(np.sum(p["dy"] * yd)) + (float(np.sum(p["dS_T"] * Sd)) if p["dS_T"] is not None else 0.0)
        lhs = float(np.sum(grads[gname] * d))
        err = abs(lhs - rhs) / max(abs(rhs), 1e-300)
        if not err < tol:
            return False, f"{gname}: <vjp,d>={lhs!r} vs <ct,jvp>={rhs!r} (rel {err:.2e})"
    return True, "ok"


def pin_strong_decay_dot_product(lib, seed=11, tol=1e-11):
    """The dot-product test with every decay in [1e-4, 1e-3] (mean log g near -8, the strong
    profile of the accuracy table in mlx issue #4614, where a chunked kernel's dg was off by
    orders of magnitude): the forward-mode side never divides by g, so a gradient that loses
    or inverts a decay factor fails here, however small the decays."""
    return pin_dot_product(lib, seed=seed, tol=tol, g_range=(1e-4, 1e-3), T=17)


# ----------------------------------------------------------------- closed forms
def pin_identity_decay_no_write(lib, seed=5, tol=1e-12):
    """g = 1, beta = 0: the state never changes. Closed forms for every output."""
    B, T, Hk, Hv, Dk, Dv = 2, 6, 2, 4, 8, 6
    p = rand_problem(seed, B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    p["g"] = np.ones((B, T, Hv))
    p["beta"] = np.zeros((B, T, Hv))
    rep = Hv // Hk
    f = run_fwd(lib, p, chunk=4)
    gr = run_bwd(lib, p, chunk=4)
    S0, dST = p["S0"], p["dS_T"]
    qh, kh = np.repeat(p["q"], rep, 2), np.repeat(p["k"], rep, 2)
    y = np.einsum("bhij,bthj->bthi", S0, qh)
    checks = {"y": (f["y"], y), "S_T": (f["S_T"], S0)}
    for c in range(f["ckpt"].shape[2]):
        checks[f"ckpt{c}"] = (f["ckpt"][:, :, c], S0)
    # Sh_t = dS_T + sum_{s >= t} dy_s q_s^T   (adjoint after adding step t's readout)
    outer = np.einsum("bthi,bthj->bthij", p["dy"], qh)
    Sh = dST[:, None] + np.flip(np.cumsum(np.flip(outer, 1), 1), 1)
    dq_h = np.einsum("bhij,bthi->bthj", S0, p["dy"])
    dd = np.einsum("bthij,bthj->bthi", Sh, kh)
    dbeta = np.einsum("bthi,bthi->bth", dd, p["v"] - np.einsum("bhij,bthj->bthi", S0, kh))
    dg = np.einsum("bthij,bhij->bth", Sh, S0)
    checks.update({
        "dq": (gr["dq"], dq_h.reshape(B, T, Hk, rep, Dk).sum(3)),
        "dk": (gr["dk"], np.zeros_like(p["k"])),
        "dv": (gr["dv"], np.zeros_like(p["v"])),
        "dg": (gr["dg"], dg), "dbeta": (gr["dbeta"], dbeta),
        "dS0": (gr["dS0"], dST + outer.sum(1)),
    })
    return _compare(checks, tol)


def pin_zero_decay(lib, seed=6, tol=1e-12):
    """g = 0: the state resets every step, S_t = beta_t v_t k_t^T (S_0 enters only step 0)."""
    B, T, Hk, Hv, Dk, Dv = 1, 7, 2, 4, 8, 6
    p = rand_problem(seed, B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, dST=False)
    p["g"] = np.zeros((B, T, Hv))
    rep = Hv // Hk
    f = run_fwd(lib, p, chunk=3)
    gr = run_bwd(lib, p, chunk=3)
    q, k, v, dy, be = np.repeat(p["q"], rep, 2), np.repeat(p["k"], rep, 2), p["v"], p["dy"], p["beta"]
    kq = np.einsum("bthj,bthj->bth", k, q)
    vdy = np.einsum("bthi,bthi->bth", v, dy)
    y = (be * kq)[..., None] * v
    dv = (be * kq)[..., None] * dy
    dbeta = kq * vdy
    dq_h = (be * vdy)[..., None] * k
    dk_h = (be * vdy)[..., None] * q
    # dg_t = beta_{t-1} (dy_t . v_{t-1}) (q_t . k_{t-1} - beta_t (q_t . k_t)(k_t . k_{t-1})), t >= 1
    dg = np.zeros((B, T, Hv))
    dg[:, 1:] = be[:, :-1] * np.einsum("bthi,bthi->bth", dy[:, 1:], v[:, :-1]) * (
        np.einsum("bthj,bthj->bth", q[:, 1:], k[:, :-1])
        - be[:, 1:] * kq[:, 1:] * np.einsum("bthj,bthj->bth", k[:, 1:], k[:, :-1]))
    # step 0 reads S_0: dg_0 = dy_0^T S0 q_0 - beta_0 (q_0.k_0) dy_0^T S0 k_0
    S0 = p["S0"]
    dg[:, 0] = (np.einsum("bhi,bhij,bhj->bh", dy[:, 0], S0, q[:, 0])
                - be[:, 0] * kq[:, 0] * np.einsum("bhi,bhij,bhj->bh", dy[:, 0], S0, k[:, 0]))
    S_T = be[:, -1, :, None, None] * np.einsum("bhi,bhj->bhij", v[:, -1], k[:, -1])
    checks = {"y": (f["y"], y), "S_T": (f["S_T"], S_T), "dv": (gr["dv"], dv),
              "dbeta": (gr["dbeta"], dbeta),
              "dq": (gr["dq"], dq_h.reshape(B, T, Hk, rep, Dk).sum(3)),
              "dk": (gr["dk"], dk_h.reshape(B, T, Hk, rep, Dk).sum(3)),
              "dg": (gr["dg"], dg), "dS0": (gr["dS0"], np.zeros_like(S0))}
    return _compare(checks, tol)


def pin_single_step(lib, seed=7, tol=1e-13):
    """T = 1: S_1 = g S0 + beta (v - g S0 k) k^T and y = S_1 q."""
    p = rand_problem(seed, B=2, T=1, Hk=1, Hv=3, Dk=5, Dv=4)
    f = run_fwd(lib, p, chunk=1)
    q, k = np.repeat(p["q"], 3, 2)[:, 0], np.repeat(p["k"], 3, 2)[:, 0]
    g, be, v, S0 = p["g"][:, 0, :, None, None], p["beta"][:, 0, :, None], p["v"][:, 0], p["S0"]
    pred = np.einsum("bhij,bhj->bhi", g * S0, k)
    S1 = g * S0 + np.einsum("bhi,bhj->bhij", be * (v - pred), k)
    y = np.einsum("bhij,bhj->bhi", S1, q)
    return _compare({"S_T": (f["S_T"], S1), "y": (f["y"][:, 0], y), "ckpt0": (f["ckpt"][:, :, 0], S0)}, tol)


def pin_orthonormal_keys(lib, seed=8, tol=1e-12):
    """Orthonormal keys and S_0 = 0: the delta term never reads anything back, and the
    recurrence is gated causal linear attention, Y = (M o (Q K^T)) diag(beta) V with
    M[t, s] = g_{s+1} ... g_t (empty product 1) for s <= t. Its q, v, g, beta gradients
    come from the matrix form by hand (reverse mode of three matrix products)."""
    B, T, Hk, Hv, Dk, Dv = 1, 6, 1, 2, 8, 5
    r = _rng(seed)
    Qm, _ = np.linalg.qr(r.standard_normal((Dk, Dk)))
    p = rand_problem(seed, B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, S0=False, dST=False)
    p["k"] = Qm[:T][None, :, None, :].copy()
    f = run_fwd(lib, p, chunk=4)
    gr = run_bwd(lib, p, chunk=4)
    q, k = p["q"][0, :, 0], p["k"][0, :, 0]
    ys, dqs = [], np.zeros_like(q)
    dgs, dbs, dvs = [], [], []
    for h in range(Hv):
        g, be, v, dy = p["g"][0, :, h], p["beta"][0, :, h], p["v"][0, :, h], p["dy"][0, :, h]
        M = np.zeros((T, T))
        for t in range(T):
            for s in range(t + 1):
                M[t, s] = np.prod(g[s + 1:t + 1])
        G = q @ k.T                     # [T, T]
        W = M * G                       # causal, gated
        ys.append(W @ (be[:, None] * v))
        # reverse mode of Y = W diag(beta) V, W = M o (Q K^T)
        dW = dy @ (be[:, None] * v).T
        dvs.append(be[:, None] * (W.T @ dy))
        dbs.append(np.einsum("si,si->s", W.T @ dy, v))
        dqs += (dW * M) @ k
        dM = dW * G
        dg = np.zeros(T)
        for t in range(T):
            for s in range(t + 1):
                for j in range(s + 1, t + 1):       # dM[t,s]/dg_j = M[t,s]/g_j without dividing
                    dg[j] += dM[t, s] * np.prod([g[i] for i in range(s + 1, t + 1) if i != j])
        dgs.append(dg)
    checks = {"y": (f["y"][0], np.stack(ys, 1)), "dv": (gr["dv"][0], np.stack(dvs, 1)),
              "dbeta": (gr["dbeta"][0], np.stack(dbs, 1)), "dg": (gr["dg"][0], np.stack(dgs, 1)),
              "dq": (gr["dq"][0, :, 0], dqs)}
    return _compare(checks, tol)


def pin_fixed_unit_key(lib, seed=9, tol=1e-12):
    """One unit key for every step, S_0 = 0, constant g and beta: S_t = x_t k^T with
    x_t = g (1 - beta) x_{t-1} + beta v_t, a first-order IIR filter (scipy.signal.lfilter)."""
    from scipy.signal import lfilter
    B, T, Hk, Hv, Dk, Dv = 1, 20, 1, 3, 6, 4
    p = rand_problem(seed, B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, S0=False, dST=False)
    kk = _rng(seed).standard_normal(Dk)
    kk /= np.linalg.norm(kk)
    p["k"] = np.broadcast_to(kk, (B, T, Hk, Dk)).copy()
    gc = np.array([0.9, 0.5, 0.99])
    bc = np.array([0.3, 0.7, 0.05])
    p["g"] = np.broadcast_to(gc, (B, T, Hv)).copy()
    p["beta"] = np.broadcast_to(bc, (B, T, Hv)).copy()
    f = run_fwd(lib, p, chunk=6)
    ys = []
    for h in range(Hv):
        x = lfilter([bc[h]], [1.0, -gc[h] * (1 - bc[h])], p["v"][0, :, h], axis=0)
        ys.append(x * (p["q"][0, :, 0] @ kk)[:, None])
    return _compare({"y": (f["y"][0], np.stack(ys, 1))}, tol)


def pin_exact_retrieval(lib, seed=10, tol=1e-12):
    """beta = 1 and unit keys: the write makes S_t k_t = v_t exactly, whatever g and S_0,
    so reading with q_t = k_t returns v_t."""
    B, T, Hk, Hv, Dk, Dv = 2, 9, 2, 4, 8, 5
    p = rand_problem(seed, B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    k = _rng(seed).standard_normal((B, T, Hk, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    p["k"], p["q"] = k, k.copy()
    p["beta"] = np.ones((B, T, Hv))
    f = run_fwd(lib, p, chunk=4)
    return _compare({"y": (f["y"], p["v"])}, tol)


def _compare(checks, tol):
    for name, (got, want) in checks.items():
        err = oracle.rel_l2(got, want) if np.linalg.norm(want) > 0 else float(np.abs(got).max())
        if not err < tol:
            return False, f"{name}: rel L2 {err:.3e} >= {tol:.1e}"
    return True, "ok"


ALL_PINS = [
    pin_finite_differences, pin_directional_fd, pin_forward_mode_jacobian, pin_dot_product,
    pin_strong_decay_dot_product,
    pin_identity_decay_no_write, pin_zero_decay, pin_single_step, pin_orthonormal_keys,
    pin_fixed_unit_key, pin_exact_retrieval,
]
