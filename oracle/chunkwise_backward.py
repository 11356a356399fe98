"""Gradient of the MDN chunkwise form, fp64 numpy (oracle, TEST INFRASTRUCTURE).

The chunk algebra a chunked gradient pass follows, for one (sequence, head)
chain, checked against the token-level reverse sweep of ``backward.py``.
Forward per chunk of n tokens (slides, frames "Solve the unknown residuals
with a lower triangular system" and "Chunk outputs combine incoming states
and local writes"; reading notes 2.4-2.5), with P = Diag(alpha) K and
Kh = Diag(eta) K:

    L    = (P Kh^T) . Gamma_m,   T = (I + L)^{-1}
    R    = V - Diag(abar_m) P S_0 + Diag(b_m) P M_0,   Vres = T R
    A    = (Q Kh^T) . Gamma
    O    = Diag(abar) Q S_0 - Diag(b) Q M_0 + A Vres
    S_n  = abar_n S_0 - b_n M_0 + [Diag(Gamma_{n,:}) Kh]^T Vres
    M_n  = mubar_n M_0 - [Diag(mu_tail) Kh]^T Vres

(``.`` the elementwise product.)  Its reverse, given dO, dS_n and dM_n:

    dVres = A^T dO + WS dS_n - WM dM_n          (WS, WM the two carry rows)
    dR    = T^T dVres;   dL = -dR Vres^T;   dV = dR
    dQ    = Diag(abar) dO S_0^T - Diag(b) dO M_0^T + (dO Vres^T . Gamma) Kh
    dS_0  = abar_n dS_n + (Diag(abar) Q)^T dO - (Diag(abar_m) P)^T dR
    dM_0  = mubar_n dM_n - b_n dS_n - (Diag(b) Q)^T dO + (Diag(b_m) P)^T dR

and dK collects the P and Kh adjoints.  dS_0, dM_0 are the adjoints at the
previous chunk's end: the chain over chunks runs backwards like the forward's
state pass runs forwards.

Gate gradients go through the chunk coefficients (Gamma, its row shift, abar,
b, their shifted copies, mu_tail and the chunk totals).  Each of these is a
sum of products in which any single gate appears at most once (Gamma_{i,j} =
sum_r beta_r prod alpha prod mu over disjoint index ranges), so it is affine
in each gate on its own, and its exact partial derivative with respect to
that gate is its value with the gate set to 1 minus its value with the gate
set to 0 (``gate_partials_by_evaluation``, the definition).
``gate_partials_closed_form`` writes the same partials as sums over Gamma's
index triangle, the form a kernel can follow.  Plus alpha's direct use in P
and eta's in Kh.  The coefficients come from ``coefficients.chunk_vectors``
(the triple-sum definition).
"""
import numpy as np

from . import coefficients as coef


def _coeffs(alpha, mu, beta):
    cv = coef.chunk_vectors(alpha, mu, beta)
    return dict(G=cv["Gamma"], Gm=cv["Gamma_m"], abar=cv["abar"], b=cv["b"],
                abar_m=cv["abar_m"], b_m=cv["b_m"], mu_tail=cv["mu_tail"],
                abar_n=cv["abar"][-1], b_n=cv["b"][-1], mubar_n=cv["mubar"][-1])


def _chunk_forward(Q, K, V, a, m, e, bt, S0, M0):
    c = _coeffs(a, m, bt)
    n = K.shape[0]
    P = a[:, None] * K
    Kh = e[:, None] * K
    X = P @ Kh.T
    T = np.linalg.inv(np.eye(n) + X * c["Gm"])
    R = V - (c["abar_m"][:, None] * P) @ S0 + (c["b_m"][:, None] * P) @ M0
    Vres = T @ R
    Y = Q @ Kh.T
    A = Y * c["G"]
    O = c["abar"][:, None] * (Q @ S0) - c["b"][:, None] * (Q @ M0) + A @ Vres
    WS = c["G"][-1, :][:, None] * Kh
    WM = c["mu_tail"][:, None] * Kh
    S_n = c["abar_n"] * S0 - c["b_n"] * M0 + WS.T @ Vres
    M_n = c["mubar_n"] * M0 - WM.T @ Vres
    saved = dict(c=c, P=P, Kh=Kh, X=X, T=T, R=R, Vres=Vres, Y=Y, A=A, WS=WS, WM=WM)
    return O, S_n, M_n, saved


def gate_partials_by_evaluation(a, m, bt, dc):
    """Gate gradients through the coefficients, one gate at a time: each
    coefficient is affine in any single gate, so its exact partial is its
    value at gate = 1 minus its value at gate = 0 (the plain definition;
    O(C^4) per chunk)."""
    gates = {"alpha": a, "mu": m, "beta": bt}
    n = len(a)
    dg = {name: np.zeros(n) for name in gates}
    for name in gates:
        for u in range(n):
            hi = {kk: vv.copy() for kk, vv in gates.items()}
            lo = {kk: vv.copy() for kk, vv in gates.items()}
            hi[name][u], lo[name][u] = 1.0, 0.0
            c1 = _coeffs(hi["alpha"], hi["mu"], hi["beta"])
            c0 = _coeffs(lo["alpha"], lo["mu"], lo["beta"])
            dg[name][u] = sum(np.sum(dc[kk] * (np.asarray(c1[kk]) - np.asarray(c0[kk])))
                              for kk in dc)
    return dg["alpha"], dg["mu"], dg["beta"]


def gate_partials_closed_form(a, m, bt, dc):
    """The same gate gradients as sums over Gamma's index triangle, without
    dividing by any gate (mu may be 0), in O(C^2) per chunk.

    Positions -1 (an origin before the chunk) and 0..n-1 (the tokens);
    A(r, i) = prod_{u=r+1}^{i} alpha_u, Mu(j, r) = prod_{u=j+1}^{r} mu_u, so
    that Gamma_{i,j} = sum_{r=max(j,0)}^{i} beta_r A(r, i) Mu(j, r), b_i is
    the origin's column, abar_i = A(-1, i), mu_tail_j = Mu(j, n-1) and
    mubar_n = Mu(-1, n-1).  With the extended adjoint dGx (the origin's
    column first) and F[i, m] = sum_{j=-1}^{m} dGx[i, j] Mu(j, m):

        dbeta_r  = sum_{i>=r} A(r, i) F[i, r]
        dalpha_u = sum_{i>=u} A(u, i) [I[i, u] + dabar_i A(-1, u-1)],
                   I[i, u] = sum_{r<u} beta_r A(r, u-1) F[i, r]
        dmu_u    = sum_{i>=u} F[i, u-1] G[i, u] + Tl_u Mu(u, n-1),
                   G[i, u] = sum_{r=u}^{i} beta_r A(r, i) Mu(u, r),
                   Tl_u = sum_{j<u} dmu_tail_j Mu(j, u-1)

    (the partial of a product is the product of its two sides of the gate).
    Each inner sum follows a one-step recurrence: F[i, m] = mu_m F[i, m-1] +
    dGx[i, m], I[i, u+1] = alpha_u I[i, u] + beta_u F[i, u], G[i, u-1] =
    beta_{u-1} A(u-1, i) + mu_u G[i, u], Tl_{u+1} = mu_u Tl_u + dmu_tail_u."""
    n = len(a)
    # product tables by multiplication only: At[r + 1, i] = A(r, i), i >= r
    At = np.zeros((n + 1, n))
    Mt = np.zeros((n + 1, n))
    for r in range(-1, n):
        pa = pm = 1.0
        if r >= 0:
            At[r + 1, r] = Mt[r + 1, r] = 1.0
        for i in range(r + 1, n):
            pa *= a[i]
            pm *= m[i]
            At[r + 1, i] = pa
            Mt[r + 1, i] = pm
    A = lambda r, i: 1.0 if i == r else At[r + 1, i]
    # fold the shifted and end copies into the base coefficients
    dG = dc["G"].copy()
    dG[:-1, :] += dc["Gm"][1:, :]
    dabar = dc["abar"].copy()
    dabar[:-1] += dc["abar_m"][1:]
    dabar[-1] += dc["abar_n"]
    db = dc["b"].copy()
    db[:-1] += dc["b_m"][1:]
    db[-1] += dc["b_n"]
    # F[i, m + 1] for m = -1..i
    F = np.zeros((n, n + 1))
    for i in range(n):
        F[i, 0] = db[i]
        for mm in range(0, i + 1):
            F[i, mm + 1] = m[mm] * F[i, mm] + dG[i, mm]
    dbeta = np.array([sum(A(r, i) * F[i, r + 1] for i in range(r, n)) for r in range(n)])
    dalpha = np.zeros(n)
    dmu = np.zeros(n)
    for i in range(n):
        inner = 0.0                                  # I[i, u]
        for u in range(0, i + 1):
            dalpha[u] += A(u, i) * (inner + dabar[i] * A(-1, u - 1))
            inner = a[u] * inner + bt[u] * F[i, u + 1]
        g = bt[i]                                    # G[i, u], u = i down to 0
        for u in range(i, -1, -1):
            dmu[u] += F[i, u] * g
            if u > 0:
                g = bt[u - 1] * A(u - 1, i) + m[u] * g
    tl = dc["mubar_n"]                               # Tl_u
    for u in range(n):
        dmu[u] += tl * (1.0 if u == n - 1 else Mt[u + 1, n - 1])
        tl = m[u] * tl + dc["mu_tail"][u]
    return dalpha, dmu, dbeta


def _chunk_backward(Q, K, V, a, m, e, bt, S0, M0, dO, dSn, dMn, sv,
                    gate_partials=gate_partials_by_evaluation):
    c, P, Kh, X, T = sv["c"], sv["P"], sv["Kh"], sv["X"], sv["T"]
    Vres, Y, A, WS, WM = sv["Vres"], sv["Y"], sv["A"], sv["WS"], sv["WM"]
    n = K.shape[0]
    dc = {name: np.zeros_like(np.asarray(val, np.float64)) for name, val in c.items()}
    # the carry
    dVres = WS @ dSn - WM @ dMn
    dWS = Vres @ dSn.T
    dWM = -Vres @ dMn.T
    dS0 = c["abar_n"] * dSn
    dM0 = -c["b_n"] * dSn + c["mubar_n"] * dMn
    dc["abar_n"] = np.sum(S0 * dSn)
    dc["b_n"] = -np.sum(M0 * dSn)
    dc["mubar_n"] = np.sum(M0 * dMn)
    dc["G"][-1, :] += np.sum(dWS * Kh, axis=1)
    dc["mu_tail"] = np.sum(dWM * Kh, axis=1)
    dKh = c["G"][-1, :][:, None] * dWS + c["mu_tail"][:, None] * dWM
    # the output
    dA = dO @ Vres.T
    dVres = dVres + A.T @ dO
    QS0, QM0 = Q @ S0, Q @ M0
    dQ = c["abar"][:, None] * (dO @ S0.T) - c["b"][:, None] * (dO @ M0.T)
    dS0 = dS0 + (c["abar"][:, None] * Q).T @ dO
    dM0 = dM0 - (c["b"][:, None] * Q).T @ dO
    dc["abar"] = np.sum(QS0 * dO, axis=1)
    dc["b"] = -np.sum(QM0 * dO, axis=1)
    dY = dA * c["G"]
    dc["G"] += dA * Y
    dQ = dQ + dY @ Kh
    dKh = dKh + dY.T @ Q
    # the residual system
    dR = T.T @ dVres
    dL = -dR @ Vres.T
    dX = dL * c["Gm"]
    dc["Gm"] = dL * X
    dP = dX @ Kh
    dKh = dKh + dX.T @ P
    dV = dR
    dPS = -dR @ S0.T          # adjoint of Diag(abar_m) P
    dPM = dR @ M0.T           # adjoint of Diag(b_m) P
    dP = dP + c["abar_m"][:, None] * dPS + c["b_m"][:, None] * dPM
    dc["abar_m"] = np.sum(P * dPS, axis=1)
    dc["b_m"] = np.sum(P * dPM, axis=1)
    dS0 = dS0 - (c["abar_m"][:, None] * P).T @ dR
    dM0 = dM0 + (c["b_m"][:, None] * P).T @ dR
    # P = Diag(alpha) K, Kh = Diag(eta) K
    dK = a[:, None] * dP + e[:, None] * dKh
    da = np.sum(dP * K, axis=1)
    de = np.sum(dKh * K, axis=1)
    # coefficients -> gates
    ga, gm, gb = gate_partials(a, m, bt, dc)
    return dict(dq=dQ, dk=dK, dv=dV, dalpha=da + ga, dmu=gm,
                deta=de, dbeta=gb), dS0, dM0


def chain_backward(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
                   do=None, dS_T=None, dM_T=None, C=64,
                   gate_partials=gate_partials_by_evaluation):
    """One chain: q, k [T, dk]; v, do [T, dv]; gates [T]; states [dk, dv].
    Gradients of <o, do> + <S_T, dS_T> + <M_T, dM_T>, chunk by chunk: the
    forward keeps each chunk's entry states, the reverse walks the chunks
    from the last, carrying the state adjoints."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, mu, eta = (np.asarray(x, np.float64).reshape(-1) for x in (alpha, mu, eta))
    T, dk = k.shape
    dv = v.shape[1]
    beta = np.ones(T) if beta is None else np.asarray(beta, np.float64).reshape(-1)
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, np.float64)
    M = np.zeros((dk, dv)) if M0 is None else np.array(M0, np.float64)
    do = np.zeros((T, dv)) if do is None else np.asarray(do, np.float64)
    dS = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T, np.float64)
    dM = np.zeros((dk, dv)) if dM_T is None else np.array(dM_T, np.float64)
    starts = list(range(0, T, C))
    entries = []
    for s0 in starts:
        sl = slice(s0, min(s0 + C, T))
        entries.append((S, M))
        _, S, M, _ = _chunk_forward(q[sl], k[sl], v[sl], alpha[sl], mu[sl],
                                    eta[sl], beta[sl], S, M)
    g = {name: np.zeros_like(x) for name, x in
         (("dq", q), ("dk", k), ("dv", v), ("dalpha", alpha), ("dmu", mu),
          ("deta", eta), ("dbeta", beta))}
    for s0, (Se, Me) in zip(reversed(starts), reversed(entries)):
        sl = slice(s0, min(s0 + C, T))
        args = (q[sl], k[sl], v[sl], alpha[sl], mu[sl], eta[sl], beta[sl], Se, Me)
        _, _, _, saved = _chunk_forward(*args)
        gc, dS, dM = _chunk_backward(*args, do[sl], dS, dM, saved, gate_partials)
        for name, val in gc.items():
            g[name][sl] = val
    g["dS0"], g["dM0"] = dS, dM
    return g


def chunk_backward_packed(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
                          do=None, dS_T=None, dM_T=None, cu_seqlens=None, C=64,
                          gate_partials=gate_partials_closed_form):
    """Packed layout (q, k [T_total, H, dk]; v, do [T_total, H, dv]; gates
    [T_total, H]; states and their adjoints [n_seq, H, dk, dv]), one chain at
    a time.  Returns the same dict as ``backward.backward``."""
    q = np.asarray(q, np.float64)
    T_total, H, dk = q.shape
    dv = np.asarray(v).shape[-1]
    cu = [0, T_total] if cu_seqlens is None else [int(c) for c in cu_seqlens]
    n_seq = len(cu) - 1
    pick = lambda x, sl, h: None if x is None else np.asarray(x, np.float64)[sl, h]
    pick_s = lambda x, s, h: None if x is None else np.asarray(x, np.float64)[s, h]
    g = {"dq": np.zeros_like(q), "dk": np.zeros((T_total, H, dk)),
         "dv": np.zeros((T_total, H, dv)), "dalpha": np.zeros((T_total, H)),
         "dmu": np.zeros((T_total, H)), "deta": np.zeros((T_total, H)),
         "dbeta": np.zeros((T_total, H)), "dS0": np.zeros((n_seq, H, dk, dv)),
         "dM0": np.zeros((n_seq, H, dk, dv))}
    for s in range(n_seq):
        sl = slice(cu[s], cu[s + 1])
        for h in range(H):
            gc = chain_backward(pick(q, sl, h), pick(k, sl, h), pick(v, sl, h),
                                pick(alpha, sl, h), pick(mu, sl, h), pick(eta, sl, h),
                                pick(beta, sl, h), pick_s(S0, s, h), pick_s(M0, s, h),
                                pick(do, sl, h), pick_s(dS_T, s, h), pick_s(dM_T, s, h),
                                C=C, gate_partials=gate_partials)
            for name in ("dq", "dk", "dv", "dalpha", "dmu", "deta", "dbeta"):
                g[name][sl, h] = gc[name]
            g["dS0"][s, h], g["dM0"][s, h] = gc["dS0"], gc["dM0"]
    return g
