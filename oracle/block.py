"""The MDN token-mixer block around the memory core, fp64 numpy (oracle, TEST
INFRASTRUCTURE: only tests/, the graft entry's smoke check and bench.py's
CPU-baseline leg use it).

The slides (frame "The memory sits inside a familiar language-model block",
Sec. 3.3 and Fig. 3 of the paper) and the reading notes (section 2.9) list
the block's steps in this order:

  1. project the input to q, k, v (per head), the output-gate input and the
     four gate projections;
  2. short causal convolution, then SiLU, on q, k and v;
  3. the Comba output correction q <- q - d k before the query is
     normalised, then L2 normalisation of q and k (``gates.prepare_qk``);
  4. the four gates from their projections (``gates.gates``);
  5. the MDN memory update (``recurrence.forward``);
  6. y_t = W_o [sigmoid(W_g x_t) * RMSNorm(o_t)].

Readings where the pages are silent (each stated where it is used):
  - the short convolution is depthwise along time, one kernel of width
    ``conv_w.shape[1]`` (4 in the workloads) per channel, causal, without
    bias, and restarts at every sequence start of a packed batch;
  - RMSNorm runs over each head's d_v outputs with a weight of d_v entries
    shared by the heads and epsilon ``eps``;
  - the projection matrix is one [d_model, 4 H d + 4 H] matrix whose columns
    are, in order, q, k, v, the output-gate input (H d each), then the
    alpha, beta, mu, eta projections (H each); W_o is [H d, d_model].
"""
import numpy as np

from . import gates as G
from . import recurrence


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def short_conv(P, w, cu_seqlens):
    """Causal depthwise convolution along the token axis: P [T_total, C],
    w [C, width] (tap j multiplies the input width - 1 - j tokens back),
    restarting at every sequence start."""
    P = np.asarray(P, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    width = w.shape[1]
    out = np.zeros_like(P)
    for s in range(len(cu_seqlens) - 1):
        a, b = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        for t in range(a, b):
            acc = np.zeros(P.shape[1])
            for j in range(width):
                src = t - (width - 1) + j
                if src >= a:
                    acc += w[:, j] * P[src]
            out[t] = acc
    return out


def rms_norm(o, weight, eps):
    """RMSNorm over the last axis: o / sqrt(mean(o^2) + eps) * weight."""
    o = np.asarray(o, dtype=np.float64)
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * np.asarray(weight, np.float64)


def block_forward(x, W_in, conv_w, rms_w, W_o, H, d, gate_params, S0=None, M0=None,
                  cu_seqlens=None, eps=1e-6, return_parts=False):
    """One MDN block on x [T_total, d_model] (packed sequences given by
    cu_seqlens, else one sequence).  gate_params: a, b, s, tau, log_mu_min,
    comba_d.  Returns (y [T_total, d_model], S_T, M_T) and, with
    return_parts, a dict of the intermediate tensors."""
    x = np.asarray(x, dtype=np.float64)
    T_total = x.shape[0]
    cu = [0, T_total] if cu_seqlens is None else [int(c) for c in cu_seqlens]
    Hd = H * d
    P = x @ np.asarray(W_in, dtype=np.float64)                          # step 1
    conv = silu(short_conv(P[:, :3 * Hd], conv_w, cu))                  # step 2
    qc = conv[:, :Hd].reshape(T_total, H, d)
    kc = conv[:, Hd:2 * Hd].reshape(T_total, H, d)
    vc = conv[:, 2 * Hd:3 * Hd].reshape(T_total, H, d)
    gp = gate_params
    q_hat, k_hat = G.prepare_qk(qc, kc, gp["comba_d"])                 # step 3
    z = [P[:, 4 * Hd + i * H:4 * Hd + (i + 1) * H] for i in range(4)]
    alpha, beta, mu, eta = G.gates(*z, a=gp["a"], b=gp["b"], s=gp["s"], tau=gp["tau"],
                                   log_mu_min=gp["log_mu_min"])        # step 4
    o, S_T, M_T = recurrence.forward(q_hat, k_hat, vc, alpha, mu, eta, beta, S0, M0,
                                     cu_seqlens=np.asarray(cu, np.int32))   # step 5
    u = 1.0 / (1.0 + np.exp(-P[:, 3 * Hd:4 * Hd])) * rms_norm(o, rms_w, eps).reshape(T_total, Hd)
    y = u @ np.asarray(W_o, dtype=np.float64)                           # step 6
    if return_parts:
        return y, S_T, M_T, dict(P=P, q_hat=q_hat, k_hat=k_hat, v=vc, alpha=alpha, beta=beta,
                                 mu=mu, eta=eta, o=o, u=u)
    return y, S_T, M_T
