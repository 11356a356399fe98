"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle on
the same inputs (all of them, or sampled independent chains), compare."""
import numpy as np
import torch

import workloads as W
from oracle import recurrence

TOL = {"fp32": 1e-4, "bf16": 2e-2}   # relative L2 per output tensor


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def gpu_chunk_fwd(x, **kw):
    import momentum_delta_rule_gb300 as mdn
    d = to_dev(x)
    o, S_T, M_T = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"],
                                d["eta"], d["beta"], d["S0"], d["M0"],
                                cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o, S_T, M_T


def chains(x):
    """List of (seq, head, token slice into the packed token axis)."""
    H = x["H"]
    if x["cu_seqlens"] is not None:
        cu = x["cu_seqlens"].tolist()
    else:
        cu = [b * x["T"] for b in range(x["B"] + 1)]
    out = []
    for s in range(len(cu) - 1):
        for h in range(H):
            out.append((s, h, slice(cu[s], cu[s + 1])))
    return out


def oracle_chains(x, sel):
    """Oracle o and final states for the selected chains.

    Returns dict chain -> (o [L, D], S_T [D, D], M_T [D, D]) in fp64.
    """
    D = x["D"]
    q = x["q"].reshape(-1, x["H"], D)
    k = x["k"].reshape(-1, x["H"], D)
    v = x["v"].reshape(-1, x["H"], D)
    g = {n: (x[n].reshape(-1, x["H"]) if x[n] is not None else None)
         for n in ("alpha", "mu", "eta", "beta")}
    res = {}
    for (s, h, sl) in sel:
        L = sl.stop - sl.start
        S0 = x["S0"][s, h][None, None] if x["S0"] is not None else None
        M0 = x["M0"][s, h][None, None] if x["M0"] is not None else None
        o, S_T, M_T = recurrence.forward(
            q[sl, h][:, None], k[sl, h][:, None], v[sl, h][:, None],
            g["alpha"][sl, h][:, None], g["mu"][sl, h][:, None],
            g["eta"][sl, h][:, None],
            None if g["beta"] is None else g["beta"][sl, h][:, None],
            S0, M0, cu_seqlens=[0, L])
        res[(s, h)] = (o[:, 0], S_T[0, 0], M_T[0, 0])
    return res


def compare(x, gpu_out, sel, tol=None):
    """Relative L2 of o, S_T and M_T over the selected chains (stacked)."""
    o, S_T, M_T = gpu_out
    tol = TOL[x["dtype"]] if tol is None else tol
    ref = oracle_chains(x, sel)
    D, H = x["D"], x["H"]
    o_flat = o.reshape(-1, H, D).float().cpu()
    got_o, ref_o, got_S, ref_S, got_M, ref_M = [], [], [], [], [], []
    for (s, h, sl) in sel:
        ro, rS, rM = ref[(s, h)]
        got_o.append(o_flat[sl, h].double().numpy())
        ref_o.append(ro)
        if S_T is not None:
            got_S.append(S_T[s, h].double().cpu().numpy())
            ref_S.append(rS)
        if M_T is not None:
            got_M.append(M_T[s, h].double().cpu().numpy())
            ref_M.append(rM)
    errs = {"o": W.rel_l2(torch.from_numpy(np.concatenate(got_o)),
                          torch.from_numpy(np.concatenate(ref_o)))}
    if got_S:
        errs["S_T"] = W.rel_l2(torch.from_numpy(np.stack(got_S)),
                               torch.from_numpy(np.stack(ref_S)))
    if got_M:
        errs["M_T"] = W.rel_l2(torch.from_numpy(np.stack(got_M)),
                               torch.from_numpy(np.stack(ref_M)))
    for key, e in errs.items():
        assert np.isfinite(e), (key, e)
        assert e <= tol, "%s rel L2 %.3e > %.1e (%s)" % (key, e, tol, errs)
    return errs
