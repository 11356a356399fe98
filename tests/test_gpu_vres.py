"""GPU parity of mdn_chunk_fwd_vres (through the C ABI): the per-token
residuals against the fp64 oracle's, and o / S_T / M_T bitwise equal to
mdn_chunk_fwd's."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import recurrence
from tests._helpers import TOL, chains, to_dev

pytestmark = pytest.mark.gpu


def _gpu(x, vres):
    import momentum_delta_rule_gb300 as mdn
    d = to_dev(x)
    out = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                        d["beta"], d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"],
                        return_vres=vres)
    torch.cuda.synchronize()
    return out


def _oracle_vres(x, sel):
    """Oracle residuals of the selected chains, stacked like the GPU's."""
    D, H = x["D"], x["H"]
    q = x["q"].reshape(-1, H, D)
    k = x["k"].reshape(-1, H, D)
    v = x["v"].reshape(-1, H, D)
    g = {n: (x[n].reshape(-1, H) if x[n] is not None else None)
         for n in ("alpha", "mu", "eta", "beta")}
    out = {}
    for (s, h, sl) in sel:
        L = sl.stop - sl.start
        S0 = x["S0"][s, h][None, None] if x["S0"] is not None else None
        M0 = x["M0"][s, h][None, None] if x["M0"] is not None else None
        res = recurrence.forward(
            q[sl, h][:, None], k[sl, h][:, None], v[sl, h][:, None],
            g["alpha"][sl, h][:, None], g["mu"][sl, h][:, None], g["eta"][sl, h][:, None],
            None if g["beta"] is None else g["beta"][sl, h][:, None],
            S0, M0, cu_seqlens=[0, L], return_vres=True)
        out[(s, h)] = res[3][:, 0]
    return out


def _check(x, sel=None):
    sel = chains(x) if sel is None else sel
    o, S_T, M_T, vres = _gpu(x, True)
    o2, S2, M2 = _gpu(x, False)
    assert torch.equal(o, o2) and torch.equal(S_T, S2) and torch.equal(M_T, M2)
    ref = _oracle_vres(x, sel)
    D, H = x["D"], x["H"]
    flat = vres.reshape(-1, H, D).double().cpu().numpy()
    got = np.concatenate([flat[sl, h] for (s, h, sl) in sel])
    want = np.concatenate([ref[(s, h)] for (s, h, sl) in sel])
    err = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err <= TOL[x["dtype"]], err
    return err


def test_vres_tiny_fp32():
    _check(W.make_prefill(W.TINY_FP32, with_beta=True))


@pytest.mark.parametrize("T", [1, 63, 65, 200])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 128)])
def test_vres_small_ragged(T, dtype, D):
    w = W.Workload("vres", dtype=dtype, state="randn", seed=21)
    _check(W.make_prefill(w, B=2, T=T, H=2, D=D, with_beta=True))


def test_vres_dual_slices():
    """Enough chains that both 64-column slices of a head share a CTA."""
    w = W.Workload("vres_dual", dtype="bf16", state="randn", seed=22)
    x = W.make_prefill(w, B=40, T=130, H=2, D=128, with_beta=True)
    _check(x, chains(x)[::5])


def test_vres_varlen_with_empty_sequences():
    _check(W.make_prefill(W.VARLEN_PACKED, H=2, lengths=[1, 64, 0, 65, 130, 7, 0]))


def test_vres_prefill_400m_full_size_sampled():
    x = W.make_prefill(W.PREFILL_400M)
    ch = chains(x)
    g = torch.Generator().manual_seed(3)
    idx = torch.randperm(len(ch), generator=g)[:3].tolist()
    _check(x, [ch[i] for i in sorted(idx)])
