"""fp64 token recurrence (oracle, test infrastructure) — Python wrapper.

The arithmetic lives in ``mdn_recurrence.c``: the MDN two-state recurrence of
the paper-reading slides ("MDN adds a momentum matrix to the delta update",
Eqs. (3)-(5)) and the reading notes, section 2.2.  This module only moves
numpy arrays in and out.

Conventions (same as the C source):
  q, k [T_total, H, dk]; v [T_total, H, dv]; gates [T_total, H];
  states [n_seq, H, dk, dv]; cu_seqlens [n_seq + 1] (host int32).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.mdn_oracle_forward.restype = ctypes.c_int
        lib.mdn_oracle_forward.argtypes = (
            [dp] * 12 + [ctypes.POINTER(ctypes.c_int32)] + [ctypes.c_int] * 5)
        lib.mdn_oracle_forward_vres.restype = ctypes.c_int
        lib.mdn_oracle_forward_vres.argtypes = (
            [dp] * 13 + [ctypes.POINTER(ctypes.c_int32)] + [ctypes.c_int] * 5)
        lib.mdn_oracle_max_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def max_threads():
    return _lib().mdn_oracle_max_threads()


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(q, k, v, alpha, mu, eta, beta=None, S0=None, M0=None,
            cu_seqlens=None, n_threads=0, return_vres=False):
    """Run the recurrence over packed sequences.

    ``q, k, v`` are ``[T_total, H, d]`` (or ``[B, T, H, d]`` with
    ``cu_seqlens=None``, meaning B equal-length sequences).  Returns
    ``(o, S_T, M_T)`` as fp64 numpy arrays; ``o`` has the shape of ``v``.
    With ``return_vres`` the residual of every token, vres_t = v_t -
    S_{t-1}^T (alpha_t k_t), comes fourth, shaped like ``v``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    alpha, mu, eta, beta = _f64(alpha), _f64(mu), _f64(eta), _f64(beta)
    S0, M0 = _f64(S0), _f64(M0)
    out_shape = v.shape
    if cu_seqlens is None:
        if q.ndim == 4:
            B, T = q.shape[0], q.shape[1]
        else:
            B, T = 1, q.shape[0]
        cu = np.arange(B + 1, dtype=np.int32) * T
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    n_seq = len(cu) - 1
    H, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    T_total = int(cu[-1])
    q = q.reshape(T_total, H, dk)
    k = k.reshape(T_total, H, dk)
    v = v.reshape(T_total, H, dv)
    gshape = (T_total, H)
    alpha = alpha.reshape(gshape)
    mu = mu.reshape(gshape)
    eta = eta.reshape(gshape)
    if beta is not None:
        beta = beta.reshape(gshape)
    sshape = (n_seq, H, dk, dv)
    if S0 is not None:
        S0 = S0.reshape(sshape)
    if M0 is not None:
        M0 = M0.reshape(sshape)
    o = np.zeros((T_total, H, dv), dtype=np.float64)
    S_T = np.zeros(sshape, dtype=np.float64)
    M_T = np.zeros(sshape, dtype=np.float64)
    vres = np.zeros((T_total, H, dv), dtype=np.float64) if return_vres else None
    rc = _lib().mdn_oracle_forward_vres(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(mu), _ptr(eta),
        _ptr(beta), _ptr(S0), _ptr(M0), _ptr(o), _ptr(S_T), _ptr(M_T), _ptr(vres),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        n_seq, H, dk, dv, int(n_threads))
    if rc != 0:
        raise RuntimeError("mdn_oracle_forward failed with code %d" % rc)
    if return_vres:
        return o.reshape(out_shape), S_T, M_T, vres.reshape(out_shape)
    return o.reshape(out_shape), S_T, M_T


def decode_step(q, k, v, alpha, mu, eta, S, M, beta=None, n_threads=0):
    """One token per sequence: ``q, k [N, H, dk]``, ``S, M [N, H, dk, dv]``.

    Returns ``(o, S_new, M_new)``; the inputs are not modified.
    """
    q = _f64(q)
    N = q.shape[0]
    o, S1, M1 = forward(q.reshape(N, 1, *q.shape[1:]),
                        _f64(k).reshape(N, 1, *q.shape[1:]),
                        _f64(v).reshape(N, 1, *_f64(v).shape[1:]),
                        _f64(alpha).reshape(N, 1, -1), _f64(mu).reshape(N, 1, -1),
                        _f64(eta).reshape(N, 1, -1),
                        None if beta is None else _f64(beta).reshape(N, 1, -1),
                        S, M, n_threads=n_threads)
    return o.reshape(_f64(v).shape), S1, M1


def default_threads():
    """Cores this process may run on (the oracle's default thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
