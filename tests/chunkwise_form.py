"""The chunkwise (dense, WY/UT) form of the gated delta rule and its VJP, in float64 numpy.

TEST INFRASTRUCTURE ONLY. This is the arithmetic a chunked tensor-core implementation would
carry out, written as plain matrix products so that its derivation can be checked against
the sequential oracle (tests/test_chunkwise_form.py). The pages do not give this form: it is
derived here from the recurrence of mlx issue #4614 ("Recurrence used for the
references"), per value head,
    S_t = g_t S_{t-1} + delta_t k_t^T,  delta_t = beta_t (v_t - g_t S_{t-1} k_t),  y_t = S_t q_t.
The same page reports that a chunked kernel returned a wrong gradient for g under strong
decay; the form below therefore never divides by g or by a cumulative decay: every decay
factor is exp of a difference of log-decay prefix sums that is <= 0, or a product of two
such factors.

Per chunk of L steps (local t = 1..L) with start state S0 [Dv, Dk]:
    lam_t = log g_t,  Lam_t = lam_1 + ... + lam_t (Lam_0 = 0),  E(s, i) = exp(Lam_s - Lam_i)
    A[t, i]  = beta_t (k_t . k_i) E(t, i)      (i < t)       T = (I + A)^-1
    R        = diag(beta) (V - diag(exp Lam) K S0^T)         Delta = T R   (rows delta_t)
    Y        = diag(exp Lam) Q S0^T + ((Q K^T) o E_incl) Delta
    S_L      = exp(Lam_L) S0 + Delta^T diag(E(L, .)) K
    U (pred) = diag(exp Lam) K S0^T + ((K K^T) o E_strict) Delta    (u_t = g_t S_{t-1} k_t)
Backward, given dY and dS_L (the adjoint of the chunk's end state):
    dD = T^T (diag(E(L, .)) K dS_L^T + ((Q K^T) o E_incl)^T dY)     (ddelta_t = Sc_t k_t)
    dU = -diag(beta) dD,  dV = diag(beta) dD,  dbeta_t = ddelta_t . (v_t - u_t)
    G = dY Delta^T,  H = dU Delta^T
    dQ = diag(exp Lam) dY S0 + (G o E_incl) K
    dK = diag(E(L, .)) Delta dS_L + (G o E_incl)^T Q + (H o E_strict)^T K
         + diag(exp Lam) dU S0 + (H o E_strict) K
    dS0 = exp(Lam_L) dS_L + dY^T diag(exp Lam) Q + dU^T diag(exp Lam) K
    dg_t = <dA_t, S_{t-1}> (dA_t = Sc_t + du_t k_t^T), expanded over the chunk's terms:
         = E(L,t) exp(Lam_{t-1}) <dS_L, S0>
         + E(L,t) sum_{i<t} E(t-1,i) f_i                       f_i = delta_i . (dS_L k_i)
         + exp(Lam_{t-1}) sum_{s>=t} E(s,t) (a_s + b_s)        a_s = dy_s . S0 q_s, b_s = du_s . S0 k_s
         + sum_{s>=t} E(s,t) sum_{i<t} E(t-1,i) W[s,i]         W = G o (Q K^T) + H o (K K^T)
      (the last term is a product of two decay-weighted L x L matrices, W times
       M[i,t] = E(t-1,i) [i < t], then a weighted column sum).
"""
from __future__ import annotations

import numpy as np


def _decay(lam):
    """Prefix sums Lam (with Lam_0 = 0 prepended) and the matrix D[s, i] = Lam_s - Lam_i."""
    Lam = np.concatenate([[0.0], np.cumsum(lam)])          # Lam[0..L]
    return Lam, Lam[:, None] - Lam[None, :]


def _rnd(x, rnd):
    return x if rnd is None else rnd(x)


def chunk_forward(S0, K, Q, V, g, beta, rnd=None):
    """One chunk of one value head. K, Q [L, Dk]; V [L, Dv]; g, beta [L]; S0 [Dv, Dk].
    `rnd`, if given, rounds every matrix-product operand (to emulate a lower-precision
    tensor-core operand type); accumulation stays float64.
    Returns Y [L, Dv], S_L [Dv, Dk], Delta [L, Dv], resid = V - U [L, Dv], and the chunk's
    intermediates (for the backward)."""
    L = K.shape[0]
    lam = np.log(g)
    Lam, Dm = _decay(lam)                  # Lam[0..L], Dm[s, i] over 0..L
    idx = np.arange(1, L + 1)
    Dloc = Dm[np.ix_(idx, idx)]            # Lam_t - Lam_i for t, i = 1..L
    tri_strict = np.tril(np.ones((L, L)), -1)
    tri_incl = np.tril(np.ones((L, L)))
    E_strict = np.exp(np.where(tri_strict > 0, Dloc, -np.inf))
    E_incl = np.exp(np.where(tri_incl > 0, Dloc, -np.inf))
    gam = np.exp(Lam[1:])                  # exp(Lam_t), t = 1..L
    eL = np.exp(Lam[L] - Lam[1:])          # E(L, t)

    KK = _rnd(K, rnd) @ _rnd(K, rnd).T
    QK = _rnd(Q, rnd) @ _rnd(K, rnd).T
    A = beta[:, None] * KK * E_strict
    T = np.linalg.inv(np.eye(L) + A)       # unit lower triangular
    KS = _rnd(K, rnd) @ _rnd(S0, rnd).T    # [L, Dv]: row t = S0 k_t
    QS = _rnd(Q, rnd) @ _rnd(S0, rnd).T
    R = beta[:, None] * (V - gam[:, None] * KS)
    Delta = _rnd(T, rnd) @ _rnd(R, rnd)
    Y = gam[:, None] * QS + _rnd(QK * E_incl, rnd) @ _rnd(Delta, rnd)
    U = gam[:, None] * KS + _rnd(KK * E_strict, rnd) @ _rnd(Delta, rnd)
    S_L = np.exp(Lam[L]) * S0 + _rnd((Delta * eL[:, None]).T, rnd) @ _rnd(K, rnd)
    ctx = dict(Lam=Lam, Dloc=Dloc, E_strict=E_strict, E_incl=E_incl, gam=gam, eL=eL, KK=KK, QK=QK,
               T=T, KS=KS, QS=QS, Delta=Delta, resid=V - U)
    return Y, S_L, Delta, V - U, ctx


def chunk_backward(S0, K, Q, V, g, beta, dY, dS_L, ctx, rnd=None):
    """VJP of one chunk (see the module docstring). Returns dQ, dK, dV, dbeta, dg, dS0."""
    L = K.shape[0]
    Lam, E_strict, E_incl = ctx["Lam"], ctx["E_strict"], ctx["E_incl"]
    gam, eL, KK, QK, T = ctx["gam"], ctx["eL"], ctx["KK"], ctx["QK"], ctx["T"]
    KS, QS, Delta, resid = ctx["KS"], ctx["QS"], ctx["Delta"], ctx["resid"]
    r = lambda x: _rnd(x, rnd)

    KdS = r(K) @ r(dS_L).T                                  # row t = dS_L k_t
    rhs = eL[:, None] * KdS + r(QK * E_incl).T @ r(dY)
    dD = r(T).T @ r(rhs)                                    # ddelta_t = Sc_t k_t
    dU = -beta[:, None] * dD
    dV = beta[:, None] * dD
    dbeta = np.sum(dD * resid, axis=1)
    G = r(dY) @ r(Delta).T                                  # G[s, i] = dy_s . delta_i
    H = r(dU) @ r(Delta).T                                  # H[s, i] = du_s . delta_i
    dQ = gam[:, None] * (r(dY) @ r(S0)) + r(G * E_incl) @ r(K)
    dK = (eL[:, None] * (r(Delta) @ r(dS_L)) + r(G * E_incl).T @ r(Q) + r(H * E_strict).T @ r(K)
          + gam[:, None] * (r(dU) @ r(S0)) + r(H * E_strict) @ r(K))
    dS0 = np.exp(Lam[L]) * dS_L + r(dY * gam[:, None]).T @ r(Q) + r(dU * gam[:, None]).T @ r(K)

    # dg_t = <dA_t, S_{t-1}>, t = 1..L, as a sum of decay-weighted terms (no division)
    LamT, LamP = Lam[1:], Lam[:-1]                          # Lam_t and Lam_{t-1}
    c0 = float(np.sum(dS_L * S0))
    f = np.sum(Delta * KdS, axis=1)                         # f_i = delta_i . (dS_L k_i)
    ab = np.sum(dY * QS, axis=1) + np.sum(dU * KS, axis=1)  # a_s + b_s
    W = G * QK + H * KK
    dg = np.empty(L)
    for t in range(L):                                      # t is the 0-based step (step t+1)
        base = Lam[L] - LamT[t] + LamP[t]
        term = np.exp(base) * c0
        i = np.arange(t)                                    # steps before t
        term += np.sum(np.exp(base - LamT[i]) * f[i])
        s = np.arange(t, L)                                 # steps at or after t
        term += np.sum(np.exp(LamP[t] + LamT[s] - LamT[t]) * ab[s])
        if t > 0:
            ex = np.exp((LamT[s] - LamT[t])[:, None] + (LamP[t] - LamT[i])[None, :])
            term += np.sum(ex * W[np.ix_(s, i)])
        dg[t] = term
    return dQ, dK, dV, dbeta, dg, dS0


def forward(q, k, v, g, beta, S0=None, chunk=64, rnd=None):
    """Whole-sequence chunkwise forward; layouts as the oracle's. Returns y, S_T, ckpt, resid."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    rep = Hv // Hk
    NC = -(-T // chunk)
    y = np.zeros((B, T, Hv, Dv))
    resid = np.zeros((B, T, Hv, Dv))
    S_T = np.zeros((B, Hv, Dv, Dk))
    ckpt = np.zeros((B, Hv, NC, Dv, Dk))
    for b in range(B):
        for h in range(Hv):
            hk = h // rep
            S = np.zeros((Dv, Dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for c in range(NC):
                t0, t1 = c * chunk, min(T, (c + 1) * chunk)
                ckpt[b, h, c] = S
                Y, S, _, R, _ = chunk_forward(S, k[b, t0:t1, hk], q[b, t0:t1, hk], v[b, t0:t1, h],
                                              g[b, t0:t1, h], beta[b, t0:t1, h], rnd)
                y[b, t0:t1, h] = Y
                resid[b, t0:t1, h] = R
            S_T[b, h] = S
    return {"y": y, "S_T": S_T, "ckpt": ckpt, "resid": resid}


def backward(q, k, v, g, beta, dy, S0=None, dS_T=None, chunk=64, rnd=None):
    """Whole-sequence chunkwise VJP (re-running each chunk's forward from its checkpoint).
    Returns dq, dk (summed over the value heads of each kv head, ascending), dv, dg, dbeta, dS0."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    rep = Hv // Hk
    NC = -(-T // chunk)
    f = forward(q, k, v, g, beta, S0, chunk, rnd)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    dg = np.zeros(g.shape)
    dbeta = np.zeros(beta.shape)
    dS0 = np.zeros((B, Hv, Dv, Dk))
    for b in range(B):
        for hk in range(Hk):
            for h in range(hk * rep, (hk + 1) * rep):
                dS = np.zeros((Dv, Dk)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
                for c in reversed(range(NC)):
                    t0, t1 = c * chunk, min(T, (c + 1) * chunk)
                    Kc, Qc, Vc = k[b, t0:t1, hk], q[b, t0:t1, hk], v[b, t0:t1, h]
                    gc, bc = g[b, t0:t1, h], beta[b, t0:t1, h]
                    S_start = f["ckpt"][b, h, c]
                    _, _, _, _, ctx = chunk_forward(S_start, Kc, Qc, Vc, gc, bc, rnd)
                    dQc, dKc, dVc, dbc, dgc, dS = chunk_backward(S_start, Kc, Qc, Vc, gc, bc, dy[b, t0:t1, h],
                                                                 dS, ctx, rnd)
                    dq[b, t0:t1, hk] += dQc
                    dk[b, t0:t1, hk] += dKc
                    dv[b, t0:t1, h] = dVc
                    dbeta[b, t0:t1, h] = dbc
                    dg[b, t0:t1, h] = dgc
                dS0[b, h] = dS
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "dS0": dS0}


# ------------------------------------------------------------------ segment scan over chunks
# The state recurrence across chunks is affine: S_L = S0 M + S_L(S0 = 0), with the chunk's state
# map M = exp(Lam_L) I - W^T diag(E(L, .)) K  [Dk, Dk],  W = T diag(beta exp Lam) K.
# A run of whole chunks (a segment) composes its chunks' maps. So the forward over NC chunks can
# run as (1) every segment from a zero start state (its end state B_j) and its composed map M_j,
# all segments independently; (2) a scan over segments, S_start(j + 1) = S_start(j) M_j + B_j;
# (3) every segment again from its true start state, independently. The VJP is linear in the
# end cotangent with the transposed map: dS_start = dS_end M^T + (the part from the segment's dy,
# D_j, its start cotangent from a zero end cotangent), so the backward scans in reverse,
# dS_end(j) = dS_end(j + 1) M_{j+1}^T + D_{j+1}, from dS_end(last) = dS_T.

def chunk_state_map(K, g, beta):
    """The chunk's state map M [Dk, Dk]: S_L = S0 M + S_L(S0 = 0)."""
    L = K.shape[0]
    Lam, Dm = _decay(np.log(g))
    idx = np.arange(1, L + 1)
    Dloc = Dm[np.ix_(idx, idx)]
    E_strict = np.exp(np.where(np.tril(np.ones((L, L)), -1) > 0, Dloc, -np.inf))
    A = beta[:, None] * (K @ K.T) * E_strict
    T = np.linalg.inv(np.eye(L) + A)
    gam = np.exp(Lam[1:])
    eL = np.exp(Lam[L] - Lam[1:])
    W = T @ ((beta * gam)[:, None] * K)
    return np.exp(Lam[L]) * np.eye(K.shape[1]) - W.T @ (eL[:, None] * K)


def segment_bounds(NC, segments):
    """Chunk index ranges [c0, c1) of `segments` runs of whole chunks (as even as possible)."""
    edges = [round(j * NC / segments) for j in range(segments + 1)]
    return [(edges[j], edges[j + 1]) for j in range(segments) if edges[j + 1] > edges[j]]


def forward_segments(q, k, v, g, beta, S0=None, chunk=64, segments=2):
    """The chunkwise forward as a scan over segments of chunks (see above). Returns y, S_T, ckpt."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    rep = Hv // Hk
    NC = -(-T // chunk)
    segs = segment_bounds(NC, segments)
    y = np.zeros((B, T, Hv, Dv))
    S_T = np.zeros((B, Hv, Dv, Dk))
    ckpt = np.zeros((B, Hv, NC, Dv, Dk))

    def run(b, h, S, c0, c1, out):
        hk = h // rep
        for c in range(c0, c1):
            t0, t1 = c * chunk, min(T, (c + 1) * chunk)
            if out:
                ckpt[b, h, c] = S
            Y, S, _, _, _ = chunk_forward(S, k[b, t0:t1, hk], q[b, t0:t1, hk], v[b, t0:t1, h], g[b, t0:t1, h],
                                          beta[b, t0:t1, h])
            if out:
                y[b, t0:t1, h] = Y
        return S

    for b in range(B):
        for h in range(Hv):
            hk = h // rep
            # (1) each segment from a zero start, and its composed map
            ends, maps = [], []
            for c0, c1 in segs:
                ends.append(run(b, h, np.zeros((Dv, Dk)), c0, c1, False))
                M = np.eye(Dk)
                for c in range(c0, c1):
                    t0, t1 = c * chunk, min(T, (c + 1) * chunk)
                    M = M @ chunk_state_map(k[b, t0:t1, hk], g[b, t0:t1, h], beta[b, t0:t1, h])
                maps.append(M)
            # (2) the scan over segments
            S = np.zeros((Dv, Dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            starts = []
            for Bj, Mj in zip(ends, maps):
                starts.append(S)
                S = S @ Mj + Bj
            S_T[b, h] = S
            # (3) each segment from its start state
            for (c0, c1), Sj in zip(segs, starts):
                run(b, h, Sj, c0, c1, True)
    return {"y": y, "S_T": S_T, "ckpt": ckpt}


def backward_segments(q, k, v, g, beta, dy, S0=None, dS_T=None, chunk=64, segments=2):
    """The chunkwise VJP as a reverse scan over segments of chunks (see above). Returns dq, dk,
    dv, dg, dbeta, dS0."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    rep = Hv // Hk
    NC = -(-T // chunk)
    segs = segment_bounds(NC, segments)
    f = forward(q, k, v, g, beta, S0, chunk)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    dg = np.zeros(g.shape)
    dbeta = np.zeros(beta.shape)
    dS0 = np.zeros((B, Hv, Dv, Dk))

    def rerun(b, h, dS, c0, c1, out):
        hk = h // rep
        for c in reversed(range(c0, c1)):
            t0, t1 = c * chunk, min(T, (c + 1) * chunk)
            Kc, Qc, Vc = k[b, t0:t1, hk], q[b, t0:t1, hk], v[b, t0:t1, h]
            gc, bc = g[b, t0:t1, h], beta[b, t0:t1, h]
            S_start = f["ckpt"][b, h, c]
            _, _, _, _, ctx = chunk_forward(S_start, Kc, Qc, Vc, gc, bc)
            dQc, dKc, dVc, dbc, dgc, dS = chunk_backward(S_start, Kc, Qc, Vc, gc, bc, dy[b, t0:t1, h], dS, ctx)
            if out:
                dq[b, t0:t1, hk] += dQc
                dk[b, t0:t1, hk] += dKc
                dv[b, t0:t1, h] = dVc
                dbeta[b, t0:t1, h] = dbc
                dg[b, t0:t1, h] = dgc
        return dS

    for b in range(B):
        for hk in range(Hk):
            for h in range(hk * rep, (hk + 1) * rep):
                # (1) each segment from a zero end cotangent, and its composed map
                locs, maps = [], []
                for c0, c1 in segs:
                    locs.append(rerun(b, h, np.zeros((Dv, Dk)), c0, c1, False))
                    M = np.eye(Dk)
                    for c in range(c0, c1):
                        t0, t1 = c * chunk, min(T, (c + 1) * chunk)
                        M = M @ chunk_state_map(k[b, t0:t1, hk], g[b, t0:t1, h], beta[b, t0:t1, h])
                    maps.append(M)
                # (2) the reverse scan over segments
                dS = np.zeros((Dv, Dk)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
                ends = [None] * len(segs)
                for j in reversed(range(len(segs))):
                    ends[j] = dS
                    dS = dS @ maps[j].T + locs[j]
                dS0[b, h] = dS
                # (3) each segment from its end cotangent
                for (c0, c1), dSj in zip(segs, ends):
                    rerun(b, h, dSj, c0, c1, True)
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "dS0": dS0}
