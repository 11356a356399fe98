"""fp64 gradient of the MDN token recurrence (oracle, TEST INFRASTRUCTURE).

The pages fix the forward only: the two-state update of the paper-reading
slides ("MDN adds a momentum matrix to the delta update", Eqs. (3)-(5)) and
the reading notes, section 2.2.  For training they add a storage policy,
not a formula (slides, "Backward computation" block beside the chunkwise
pseudocode; reading notes, end of section 2.6; slides frame "Training speed
improves when residuals are saved"): keep the residuals vres_t from the
forward, rebuild the states from them for the gradient, and do not keep
every (S, M) pair.  So the gradient here is the plain definition: the
vector-Jacobian product of the forward, taken one token at a time in reverse,
with the states rebuilt from the chunk-entry states and the saved residuals
as that block describes (``rebuild_states``).

Per token, with S', M' the states after the token and S, M those before:

    p    = alpha k;  vres = v - S^T p
    M'   = mu M - eta k vres^T
    S'   = alpha S - beta M'
    o    = S'^T q

Given the adjoints do, dS' and dM' (dS' already holding every later
token's contribution), the reverse step is

    dq   = S' do;                 dS' += q do^T
    dalpha = <S, dS'>;            dbeta = -<M', dS'>
    dM'' = dM' - beta dS'         (the full adjoint of M')
    dmu  = <M, dM''>;             deta = -k^T dM'' vres
    dk   = -eta dM'' vres;        dvres = -eta dM''^T k
    dv   = dvres
    dS   = alpha dS' - p dvres^T; dM = mu dM''
    dalpha += -k^T S dvres;       dk += -alpha S dvres

Layouts follow the forward oracle: q, k [T_total, H, dk]; v, do
[T_total, H, dv]; gates [T_total, H]; states [n_seq, H, dk, dv];
cu_seqlens [n_seq + 1].  Pure numpy, one token at a time, all heads at once:
for the small cases of the tests.
"""
import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def rebuild_states(k, alpha, mu, eta, beta, vres, S_entry, M_entry):
    """States after every token of one segment, from its entry states and the
    saved residuals alone (no S^T k product): M' = mu M - eta k vres^T and
    S' = alpha S - beta M'.

    k [n, H, dk]; vres [n, H, dv]; gates [n, H]; S_entry, M_entry [H, dk, dv].
    Returns S_all, M_all [n + 1, H, dk, dv], index 0 the entry states."""
    k, vres = _f64(k), _f64(vres)
    alpha, mu, eta = _f64(alpha), _f64(mu), _f64(eta)
    n, H = k.shape[0], k.shape[1]
    beta = np.ones((n, H)) if beta is None else _f64(beta)
    S = np.array(_f64(S_entry), copy=True)
    M = np.array(_f64(M_entry), copy=True)
    S_all = np.empty((n + 1,) + S.shape)
    M_all = np.empty((n + 1,) + M.shape)
    S_all[0], M_all[0] = S, M
    for t in range(n):
        M = mu[t][:, None, None] * M - eta[t][:, None, None] * np.einsum("hi,hj->hij", k[t], vres[t])
        S = alpha[t][:, None, None] * S - beta[t][:, None, None] * M
        S_all[t + 1], M_all[t + 1] = S, M
    return S_all, M_all


def _residuals(k, v, alpha, S_before):
    """vres_t = v_t - S_{t-1}^T (alpha_t k_t) for every token of a segment."""
    p = alpha[:, :, None] * k
    return v - np.einsum("thij,thi->thj", S_before, p)


def backward(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
             do=None, dS_T=None, dM_T=None, cu_seqlens=None):
    """Gradients of  <o, do> + <S_T, dS_T> + <M_T, dM_T>  with respect to
    every input of the forward.  None for do / dS_T / dM_T means zero; None
    for S0 / M0 means zero initial states; None for beta means beta = 1 (its
    gradient at 1 is still returned).

    Returns a dict with dq, dk, dv, dalpha, dmu, deta, dbeta, dS0, dM0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    alpha, mu, eta = _f64(alpha), _f64(mu), _f64(eta)
    Tt, H, dk = q.shape
    dv_ = v.shape[2]
    beta = np.ones((Tt, H)) if beta is None else _f64(beta)
    cu = np.asarray([0, Tt] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    n_seq = len(cu) - 1
    zeros_state = np.zeros((n_seq, H, dk, dv_))
    S0 = zeros_state if S0 is None else _f64(S0)
    M0 = zeros_state if M0 is None else _f64(M0)
    do = np.zeros((Tt, H, dv_)) if do is None else _f64(do)
    dS_T = zeros_state if dS_T is None else _f64(dS_T)
    dM_T = zeros_state if dM_T is None else _f64(dM_T)

    g = {name: np.zeros_like(x) for name, x in
         (("dq", q), ("dk", k), ("dv", v), ("dalpha", alpha), ("dmu", mu),
          ("deta", eta), ("dbeta", beta))}
    g["dS0"] = np.zeros((n_seq, H, dk, dv_))
    g["dM0"] = np.zeros((n_seq, H, dk, dv_))

    for s in range(n_seq):
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        # the forward, keeping only the residuals; the states the reverse
        # sweep needs are then rebuilt from them and the entry states
        vres = np.empty((n, H, dv_))
        S = S0[s].copy()
        M = M0[s].copy()
        for t in range(n):
            vres[t] = _residuals(k[a + t:a + t + 1], v[a + t:a + t + 1],
                                 alpha[a + t:a + t + 1], S[None])[0]
            M = mu[a + t][:, None, None] * M - eta[a + t][:, None, None] * np.einsum(
                "hi,hj->hij", k[a + t], vres[t])
            S = alpha[a + t][:, None, None] * S - beta[a + t][:, None, None] * M
        S_all, M_all = rebuild_states(k[a:b], alpha[a:b], mu[a:b], eta[a:b],
                                      beta[a:b], vres, S0[s], M0[s])

        dS = dS_T[s].copy()
        dM = dM_T[s].copy()
        for t in range(n - 1, -1, -1):
            i = a + t
            Sb, Mb = S_all[t], M_all[t]            # before the token
            Sa, Ma = S_all[t + 1], M_all[t + 1]    # after it
            al, m_, be = (x[i][:, None, None] for x in (alpha, mu, beta))
            # o = S'^T q
            g["dq"][i] = np.einsum("hij,hj->hi", Sa, do[i])
            dS = dS + np.einsum("hi,hj->hij", q[i], do[i])
            # S' = alpha S - beta M'
            g["dalpha"][i] = np.einsum("hij,hij->h", Sb, dS)
            g["dbeta"][i] = -np.einsum("hij,hij->h", Ma, dS)
            dMf = dM - be * dS
            # M' = mu M - eta k vres^T
            g["dmu"][i] = np.einsum("hij,hij->h", Mb, dMf)
            g["deta"][i] = -np.einsum("hi,hij,hj->h", k[i], dMf, vres[t])
            dkt = -eta[i][:, None] * np.einsum("hij,hj->hi", dMf, vres[t])
            dvres = -eta[i][:, None] * np.einsum("hij,hi->hj", dMf, k[i])
            # vres = v - S^T (alpha k)
            g["dv"][i] = dvres
            p = alpha[i][:, None] * k[i]
            S_dvres = np.einsum("hij,hj->hi", Sb, dvres)
            g["dalpha"][i] += -np.einsum("hi,hi->h", k[i], S_dvres)
            g["dk"][i] = dkt - alpha[i][:, None] * S_dvres
            dS = al * dS - np.einsum("hi,hj->hij", p, dvres)
            dM = m_ * dMf
        g["dS0"][s] = dS
        g["dM0"][s] = dM
    return g
