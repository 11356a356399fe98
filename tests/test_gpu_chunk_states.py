"""GPU parity of the per-chunk entry states (mdn_chunk_fwd_states): for
chunk c of every sequence, the states after its first 64 c tokens, against
the oracle recurrence run chunk by chunk from the previous chunk's states
(split-sequence state passing, which the oracle's own tests pin).  Covers
tensor-core slices of 16 and 64 columns, fp32 inputs (split operands) and
head size 64, ragged last chunks, packed sequences with empty
members, mu = 0 entries and nonzero initial states.  The states are stored
in the input precision (bf16 for bf16 inputs), so chunk 0 holds the
initial states rounded to it."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import recurrence
from oracle import backward as bwd
from tests._helpers import TOL, chains, oracle_chains, to_dev

pytestmark = pytest.mark.gpu
C = 64


def _oracle_chunk_states(x, s, h, sl):
    D, H = x["D"], x["H"]
    sel = lambda n: x[n].reshape(-1, H, D)[sl, h] if n in ("q", "k", "v") else (
        None if x[n] is None else x[n].reshape(-1, H)[sl, h])
    q, k, v = sel("q"), sel("k"), sel("v")
    a, mu, eta, beta = sel("alpha"), sel("mu"), sel("eta"), sel("beta")
    S = x["S0"][s, h].double().numpy() if x["S0"] is not None else np.zeros((D, D))
    M = x["M0"][s, h].double().numpy() if x["M0"] is not None else np.zeros((D, D))
    L = sl.stop - sl.start
    nch = (L + C - 1) // C
    out = []
    for c in range(nch):
        out.append((S, M))
        if c == nch - 1:
            break
        seg = slice(c * C, (c + 1) * C)
        _, S_T, M_T = recurrence.forward(
            q[seg][:, None], k[seg][:, None], v[seg][:, None], a[seg][:, None],
            mu[seg][:, None], eta[seg][:, None],
            None if beta is None else beta[seg][:, None],
            torch.from_numpy(S)[None, None], torch.from_numpy(M)[None, None],
            cu_seqlens=[0, C])
        S, M = S_T[0, 0], M_T[0, 0]
    return out


def _check(x, max_chains=None):
    import momentum_delta_rule_gb300 as mdn
    d = to_dev(x)
    o, S_T, M_T, Sc, Mc = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"],
                                        d["eta"], d["beta"], d["S0"], d["M0"],
                                        cu_seqlens=d["cu_seqlens"], return_chunk_states=True)
    o2, S2, M2 = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                               d["beta"], d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    tol = TOL[x["dtype"]]
    # the forward's own results are those of the plain call
    for a_, b_ in ((o, o2), (S_T, S2), (M_T, M2)):
        a_, b_ = a_.double(), b_.double()
        assert ((a_ - b_).norm() / b_.norm().clamp_min(1e-30)).item() <= tol * 1e-2
    sdt = torch.bfloat16 if x["dtype"] == "bf16" else torch.float32
    assert Sc.dtype == sdt and Mc.dtype == sdt
    Sc, Mc = Sc.double().cpu().numpy(), Mc.double().cpu().numpy()
    ch = chains(x)
    if max_chains is not None:
        ch = ch[:: max(1, len(ch) // max_chains)]
    lens = [c.stop - c.start for (_, h, c) in chains(x) if h == 0]
    slot0 = np.concatenate([[0], np.cumsum([(L + C - 1) // C for L in lens])])
    got, want = [], []
    for (s, h, sl) in ch:
        ref = _oracle_chunk_states(x, s, h, sl)
        for c, (rS, rM) in enumerate(ref):
            got.append(np.stack([Sc[slot0[s] + c, h], Mc[slot0[s] + c, h]]))
            want.append(np.stack([rS, rM]))
        if ref:
            # chunk 0 carries the initial states (rounded to the storage type)
            S0 = x["S0"][s, h].to(sdt).double().numpy() if x["S0"] is not None else 0.0
            assert np.array_equal(Sc[slot0[s], h], np.broadcast_to(S0, Sc[slot0[s], h].shape))
    got, want = np.stack(got), np.stack(want)
    err = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert err <= tol, err


def test_chunk_states_ragged_narrow_slices():
    w = W.Workload("cs_ragged", dtype="bf16", state="randn", seed=51)
    x = W.make_prefill(w, B=3, T=130, H=4, D=128, with_beta=True)
    x["mu"][:, ::5] = 0.0
    _check(x)


def test_chunk_states_wide_slices():
    w = W.Workload("cs_wide", dtype="bf16", state="randn", seed=52)
    x = W.make_prefill(w, B=3, T=150, H=16, D=128, with_beta=True)
    _check(x, max_chains=8)


def test_chunk_states_packed_with_empty_sequences():
    x = W.make_prefill(W.VARLEN_PACKED, H=4, lengths=[1, 64, 0, 65, 130, 7], seed=53)
    _check(x)


def test_chunk_states_dual_slices():
    """Enough chains that both 64-column slices of a head share a CTA."""
    w = W.Workload("cs_dual", dtype="bf16", state="randn", seed=55)
    x = W.make_prefill(w, B=40, T=130, H=2, D=128, with_beta=True)
    _check(x, max_chains=10)


@pytest.mark.parametrize("dtype,D", [("fp32", 64), ("fp32", 128), ("bf16", 64)])
def test_chunk_states_split_and_head_size_64(dtype, D):
    w = W.Workload("cs_fp32", dtype=dtype, state="randn", seed=54)
    x = W.make_prefill(w, B=2, T=130, H=2, D=D, with_beta=True)
    _check(x)


def test_states_rebuilt_from_saved_residuals():
    """What a gradient pass keeps (slides, "Backward computation" block: save
    the residuals, rebuild the states): each chunk's states rebuilt from the
    forward's saved entry states and saved residuals, by M' = mu M -
    eta k vres^T and S' = alpha S - beta M', match the oracle's states at the
    next chunk boundary and at the sequence end (ragged last chunk, mu = 0
    entries, nonzero initial states)."""
    import momentum_delta_rule_gb300 as mdn
    w = W.Workload("cs_rebuild", dtype="bf16", state="randn", seed=55)
    x = W.make_prefill(w, B=2, T=150, H=2, D=128, with_beta=True)
    x["mu"][:, ::7] = 0.0
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], d["beta"],
            d["S0"], d["M0"])
    _, _, _, Sc, Mc = mdn.chunk_fwd(*args, return_chunk_states=True)
    _, _, _, vres = mdn.chunk_fwd(*args, return_vres=True)
    torch.cuda.synchronize()
    Sc, Mc = Sc.double().cpu().numpy(), Mc.double().cpu().numpy()
    D, H = x["D"], x["H"]
    vres = vres.double().cpu().numpy().reshape(-1, H, D)
    k = x["k"].double().numpy().reshape(-1, H, D)
    g = {n: x[n].double().numpy().reshape(-1, H) for n in ("alpha", "mu", "eta", "beta")}
    ch = chains(x)
    finals = oracle_chains(x, ch)
    lens = [c.stop - c.start for (_, h, c) in ch if h == 0]
    slot0 = np.concatenate([[0], np.cumsum([(L + C - 1) // C for L in lens])])
    got, want = [], []
    for (s, h, sl) in ch:
        L = sl.stop - sl.start
        ref = _oracle_chunk_states(x, s, h, sl)
        nch = (L + C - 1) // C
        slot = slot0[s]
        for c in range(nch):
            seg = slice(sl.start + c * C, sl.start + min((c + 1) * C, L))
            S_all, M_all = bwd.rebuild_states(
                k[seg, h][:, None], g["alpha"][seg, h][:, None], g["mu"][seg, h][:, None],
                g["eta"][seg, h][:, None], g["beta"][seg, h][:, None],
                vres[seg, h][:, None], Sc[slot + c, h][None], Mc[slot + c, h][None])
            target = ref[c + 1] if c + 1 < nch else finals[(s, h)][1:]
            got.append(np.stack([S_all[-1, 0], M_all[-1, 0]]))
            want.append(np.stack([target[0], target[1]]))
    got, want = np.stack(got), np.stack(want)
    err = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert err <= TOL["bf16"], err
