"""Chunk coefficients of the MDN chunkwise form, fp64 (oracle, test only).

Inside one chunk, tokens are numbered 1..C (index r-1 in the arrays) and the
chunk's entry states are S_0, M_0.  The pages define, for j <= i,

  abar_i = prod_{r<=i} alpha_r,  mubar_i = prod_{r<=i} mu_r,
  c_i    = sum_{r<=i} beta_r mubar_r / abar_r,   b_i = abar_i c_i,
  gamma_{i,j} = (abar_i / mubar_j) (c_i - c_{j-1})
              = sum_{r=j}^{i} beta_r prod_{u=r+1}^{i} alpha_u prod_{u=j+1}^{r} mu_u

(slides, frame "Reorder the triangular sum to isolate scalar coefficients",
Eqs. (7)-(9) and Appendix C Eqs. (30)-(31); reading notes section 2.3).
The log-domain statement of Algorithm 1 is in the slides' backup frame "use
the consistent log-domain coefficients" and in reading notes section 2.6.

Four independent evaluations are provided so the tests can play them against
each other:

  gamma_triple_sum   the explicit triple-product sum (the definition)
  gamma_cumulative   the cumulative-product / c_i form (Eqs. (7)-(9))
  gamma_printed_log  the printed log-domain form; it cancels catastrophically
                     once l_i - l_{j-1} drops below the working precision, so
                     it is only trusted on well-conditioned gates
  gamma_column_recurrence
                     gamma_{i,j} = alpha_i gamma_{i-1,j} + beta_i prod_{u=j+1}^{i} mu_u,
                     gamma_{j,j} = beta_j  (every term non-negative)

Each returns ``(Gamma, b)`` with ``Gamma`` the C x C lower-triangular matrix
(zero above the diagonal) and ``b`` the length-C vector b_1..b_C.
"""
import numpy as np


def _as1d(x):
    return np.asarray(x, dtype=np.float64).reshape(-1)


def gamma_triple_sum(alpha, mu, beta):
    alpha, mu, beta = _as1d(alpha), _as1d(mu), _as1d(beta)
    C = alpha.shape[0]
    G = np.zeros((C, C))
    b = np.zeros(C)
    for i in range(C):
        for j in range(i + 1):
            s = 0.0
            for r in range(j, i + 1):
                s += beta[r] * np.prod(alpha[r + 1:i + 1]) * np.prod(mu[j + 1:r + 1])
            G[i, j] = s
        # b_i: the same sum with the error's origin before the chunk (j = 0,
        # mubar_0 = 1), i.e. every mu_1..mu_r multiplies in.
        s = 0.0
        for r in range(0, i + 1):
            s += beta[r] * np.prod(alpha[r + 1:i + 1]) * np.prod(mu[0:r + 1])
        b[i] = s
    return G, b


def gamma_cumulative(alpha, mu, beta):
    alpha, mu, beta = _as1d(alpha), _as1d(mu), _as1d(beta)
    C = alpha.shape[0]
    abar = np.cumprod(alpha)
    mubar = np.cumprod(mu)
    c = np.cumsum(beta * mubar / abar)
    b = abar * c
    G = np.zeros((C, C))
    for i in range(C):
        for j in range(i + 1):
            c_prev = c[j - 1] if j >= 1 else 0.0
            G[i, j] = abar[i] / mubar[j] * (c[i] - c_prev)
    return G, b


def gamma_printed_log(alpha, mu, beta):
    alpha, mu, beta = _as1d(alpha), _as1d(mu), _as1d(beta)
    C = alpha.shape[0]
    with np.errstate(divide="ignore"):
        A = np.cumsum(np.log(alpha))
        U = np.cumsum(np.log(mu))
        x = np.log(beta) + U - A
    ell = np.logaddexp.accumulate(x)            # logcumsumexp, ell_0 = -inf
    b = np.exp(A + ell)
    G = np.zeros((C, C))
    for i in range(C):
        for j in range(i + 1):
            ell_prev = ell[j - 1] if j >= 1 else -np.inf
            G[i, j] = np.exp(A[i] + ell[i] - U[j]) * (1.0 - np.exp(ell_prev - ell[i]))
    return G, b


def gamma_column_recurrence(alpha, mu, beta):
    alpha, mu, beta = _as1d(alpha), _as1d(mu), _as1d(beta)
    C = alpha.shape[0]
    G = np.zeros((C, C))
    b = np.zeros(C)
    for j in range(C):
        m = 1.0                                 # prod_{u=j+1}^{i} mu_u
        g = beta[j]                             # gamma_{j,j} = beta_j
        G[j, j] = g
        for i in range(j + 1, C):
            m *= mu[i]
            g = alpha[i] * g + beta[i] * m
            G[i, j] = g
    m = 1.0                                     # mubar_i for b
    g = 0.0
    for i in range(C):
        m *= mu[i]
        g = alpha[i] * g + beta[i] * m
        b[i] = g
    return G, b


def chunk_vectors(alpha, mu, beta, gamma_fn=gamma_triple_sum):
    """All per-chunk coefficient objects the chunkwise form uses.

    Returns a dict with
      Gamma    C x C, gamma_{i,j} on and below the diagonal
      Gamma_m  the row-shifted Gamma: Gamma_m[i, j] = gamma_{i-1, j} for j < i,
               first row zero (slides backup "a one-row shift is essential")
      abar, mubar, b           length C
      abar_m   (1, abar_1, ..., abar_{C-1})
      b_m      (0, b_1, ..., b_{C-1})
      mu_tail  prod_{u=j+1}^{C} mu_u  (= mubar_C / mubar_j, no division)
    """
    alpha, mu, beta = _as1d(alpha), _as1d(mu), _as1d(beta)
    C = alpha.shape[0]
    G, b = gamma_fn(alpha, mu, beta)
    Gm = np.zeros((C, C))
    Gm[1:, :] = G[:-1, :]
    abar = np.cumprod(alpha)
    mubar = np.cumprod(mu)
    abar_m = np.concatenate([[1.0], abar[:-1]])
    b_m = np.concatenate([[0.0], b[:-1]])
    mu_tail = np.array([np.prod(mu[j + 1:]) for j in range(C)])
    return dict(Gamma=G, Gamma_m=Gm, abar=abar, mubar=mubar, b=b,
                abar_m=abar_m, b_m=b_m, mu_tail=mu_tail)
