"""MDN chunkwise-parallel forward, fp64 numpy (oracle, test only).

Follows the pages' chunk algebra step by step for one (sequence, head) chain:

  slides, frames "Reorder the triangular sum ..." (Eqs. (7)-(9)),
  "Solve the unknown residuals with a lower triangular system"
  (Eqs. (15)-(18)), "Chunk outputs combine incoming states and local writes"
  (Appendix C Eqs. (40)-(42)), backup "a one-row shift is essential";
  reading notes sections 2.3-2.5.

Per chunk of C tokens (rows stacked), with khat_j = eta_j k_j, p_i = alpha_i k_i:

  T     = [I + (P Khat^T) . Gamma_m]^{-1}
  U     = T V,  Y = T Diag(abar_m) P,  Z = T Diag(b_m) P
  Vres  = U - Y S_0 + Z M_0
  O     = Diag(abar) Q S_0 - Diag(b) Q M_0 + [(Q Khat^T) . Gamma] Vres
  S_nxt = abar_C S_0 - b_C M_0 + [Diag(Gamma_{C,:}) Khat]^T Vres
  M_nxt = mubar_C M_0 - [Diag(mubar_C / mubar) Khat]^T Vres

(``.`` is the elementwise product.)  A library solve serves as the inverse.
A final chunk shorter than C uses its own length (each sequence is chunked
from its own start).

``shift`` selects the matrix in the residual system: ``"row"`` (the pages'
row-shifted Gamma, correct) or ``"strict"`` (Gamma with its diagonal deleted —
the mistake the backup slide warns about; kept only so a test can show that
the pins catch it).
"""
import numpy as np

from . import coefficients as coef


def chunk_forward(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
                  C=64, gamma_fn=coef.gamma_triple_sum, shift="row",
                  return_vres=False):
    """One chain: ``q, k [T, dk]``, ``v [T, dv]``, gates ``[T]``.

    Returns ``(o [T, dv], S_T, M_T)`` (and the residuals Vres [T, dv] when
    ``return_vres``).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    alpha = np.asarray(alpha, np.float64).reshape(-1)
    mu = np.asarray(mu, np.float64).reshape(-1)
    eta = np.asarray(eta, np.float64).reshape(-1)
    T, dk = k.shape
    dv = v.shape[1]
    beta = np.ones(T) if beta is None else np.asarray(beta, np.float64).reshape(-1)
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, np.float64)
    M = np.zeros((dk, dv)) if M0 is None else np.array(M0, np.float64)
    o = np.zeros((T, dv))
    vres_all = np.zeros((T, dv))

    for start in range(0, T, C):
        end = min(start + C, T)
        sl = slice(start, end)
        a, m, e, bt = alpha[sl], mu[sl], eta[sl], beta[sl]
        Q, K, V = q[sl], k[sl], v[sl]
        cv = coef.chunk_vectors(a, m, bt, gamma_fn)
        G = cv["Gamma"]
        if shift == "row":
            Gm = cv["Gamma_m"]
        elif shift == "strict":
            Gm = np.tril(G, -1)
        else:
            raise ValueError(shift)
        P = a[:, None] * K
        Khat = e[:, None] * K
        n = end - start
        T_mat = np.linalg.inv(np.eye(n) + (P @ Khat.T) * Gm)
        U = T_mat @ V
        Y = T_mat @ (cv["abar_m"][:, None] * P)
        Z = T_mat @ (cv["b_m"][:, None] * P)
        Vres = U - Y @ S + Z @ M
        O = (cv["abar"][:, None] * (Q @ S) - cv["b"][:, None] * (Q @ M)
             + ((Q @ Khat.T) * G) @ Vres)
        S_next = (cv["abar"][-1] * S - cv["b"][-1] * M
                  + (G[-1, :][:, None] * Khat).T @ Vres)
        M_next = cv["mubar"][-1] * M - (cv["mu_tail"][:, None] * Khat).T @ Vres
        S, M = S_next, M_next
        o[sl] = O
        vres_all[sl] = Vres
    if return_vres:
        return o, S, M, vres_all
    return o, S, M


def chunk_forward_packed(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
                         cu_seqlens=None, C=64, **kw):
    """Packed layout ``[T_total, H, d]`` with ``cu_seqlens``; chains in a loop."""
    q = np.asarray(q, np.float64)
    T_total, H, dk = q.shape
    dv = np.asarray(v).shape[-1]
    if cu_seqlens is None:
        cu_seqlens = [0, T_total]
    cu = [int(x) for x in cu_seqlens]
    n_seq = len(cu) - 1
    o = np.zeros((T_total, H, dv))
    S_T = np.zeros((n_seq, H, dk, dv))
    M_T = np.zeros((n_seq, H, dk, dv))
    for s in range(n_seq):
        sl = slice(cu[s], cu[s + 1])
        for h in range(H):
            o_, S_, M_ = chunk_forward(
                q[sl, h], np.asarray(k)[sl, h], np.asarray(v)[sl, h],
                np.asarray(alpha)[sl, h], np.asarray(mu)[sl, h],
                np.asarray(eta)[sl, h],
                None if beta is None else np.asarray(beta)[sl, h],
                None if S0 is None else np.asarray(S0)[s, h],
                None if M0 is None else np.asarray(M0)[s, h], C=C, **kw)
            o[sl, h] = o_
            S_T[s, h] = S_
            M_T[s, h] = M_
    return o, S_T, M_T
