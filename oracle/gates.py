"""Gate parameterisation and query/key preparation of an MDN layer, fp64
(oracle, test infrastructure only; only tests/, the graft entry's smoke check
and bench.py's CPU-baseline leg use it).

Gates, per token and head, from the scalar projections z = W x_t (slides,
frame "Coupled gates restrict the spectral region", Sec. 3.3; reading notes
section 2.8):

  eta_t   = 1 + tanh(z_eta / tau)                       in (0, 2)
  theta_t = arctan(s eta_t)
  alpha_max = cos^2 theta_t,  beta_max = sin^2 theta_t   (sum to 1)
  log alpha_t = f(z_alpha) + log alpha_max
  beta_t      = sigmoid(z_beta) beta_max
  log mu_t    = max(f(z_mu), log_mu_min)
  f(z) = -a softplus(z + b)

so alpha_t + beta_t <= 1.  The reported experiments use log_mu_min = -2.

Queries and keys (reading notes section 2.9, Fig. 3 of the paper): the
layer's output correction from Comba subtracts d k_t from the query before
the query is normalised; both are then L2-normalised per head.  Reading
taken here: the correction uses the key at the same stage (before its own
normalisation), and a row of norm zero stays zero.
"""
import numpy as np


def softplus(x):
    x = np.asarray(x, dtype=np.float64)
    return np.logaddexp(0.0, x)


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def gates(z_alpha, z_beta, z_mu, z_eta, a, b, s, tau, log_mu_min):
    """Return (alpha, beta, mu, eta) as fp64 arrays shaped like the inputs."""
    za, zb, zm, ze = (np.asarray(z, dtype=np.float64) for z in (z_alpha, z_beta, z_mu, z_eta))
    eta = 1.0 + np.tanh(ze / tau)
    theta = np.arctan(s * eta)
    alpha_max = np.cos(theta) ** 2
    beta_max = np.sin(theta) ** 2
    f = lambda z: -a * softplus(z + b)
    log_alpha = f(za) + np.log(alpha_max)
    beta = sigmoid(zb) * beta_max
    log_mu = np.maximum(f(zm), log_mu_min)
    return np.exp(log_alpha), beta, np.exp(log_mu), eta


def _l2_rows(x):
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)


def prepare_qk(q, k, comba_d):
    """q, k [..., d] -> (q_hat, k_hat): q_hat = (q - d k) / |q - d k|,
    k_hat = k / |k| (fp64)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    return _l2_rows(q - comba_d * k), _l2_rows(k)
