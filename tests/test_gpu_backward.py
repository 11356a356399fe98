"""GPU parity of the gradient pass (mdn_chunk_bwd, through the C ABI) against
the fp64 token-level oracle (oracle/backward.py, itself pinned to central
differences of the forward oracle).

The forward's chunk entry states come from mdn_chunk_fwd_states on the GPU,
as a training step would use them.  Every gradient (q, k, v, the four gates,
the initial states) is compared by relative L2 over the compared chains at
the forward's tolerances: 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.
Small cases compare every chain; the full-size workloads compare sampled
(sequence, head) chains, each against a full oracle run of that chain.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import backward as bwd
from tests._helpers import TOL, chains, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dalpha", "dmu", "deta", "dbeta", "dS0", "dM0")


def _adjoints(x, seed, with_state_adjoints=True):
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(x["v"].shape, generator=g).to(x["v"].dtype)
    n_seq, H, D = x["n_seq"], x["H"], x["D"]
    if not with_state_adjoints:
        return do, None, None
    dS = torch.randn((n_seq, H, D, D), generator=g) * 0.1
    dM = torch.randn((n_seq, H, D, D), generator=g) * 0.1
    return do, dS, dM


def _gpu_grads(x, do, dS, dM):
    import momentum_delta_rule_gb300 as mdn
    d = to_dev(x)
    _, _, _, Sc, Mc = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                                    d["beta"], d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"],
                                    return_chunk_states=True)
    g = mdn.chunk_bwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], Sc, Mc,
                      do.cuda(), beta=d["beta"],
                      dS_T=None if dS is None else dS.cuda(),
                      dM_T=None if dM is None else dM.cuda(),
                      cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert mdn.device_status() == mdn.MDN_OK
    return {k: (None if v is None else v.cpu()) for k, v in g.items()}


def _oracle_chain(x, do, dS, dM, s, h, sl):
    D, H = x["D"], x["H"]
    pick = lambda t: t.reshape(-1, H, D)[sl, h:h + 1]
    pick_g = lambda t: None if t is None else t.reshape(-1, H)[sl, h:h + 1]
    st = lambda t: None if t is None else t[s:s + 1, h:h + 1]
    return bwd.backward(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick_g(x["alpha"]),
                        pick_g(x["mu"]), pick_g(x["eta"]), pick_g(x["beta"]),
                        st(x["S0"]), st(x["M0"]), pick(do), st(dS), st(dM),
                        cu_seqlens=[0, sl.stop - sl.start])


def _compare(x, got, do, dS, dM, sel, tol=None):
    tol = TOL[x["dtype"]] if tol is None else tol
    D, H = x["D"], x["H"]
    acc = {n: ([], []) for n in NAMES}
    for (s, h, sl) in sel:
        ref = _oracle_chain(x, do, dS, dM, s, h, sl)
        for n in ("dq", "dk", "dv"):
            acc[n][0].append(got[n].reshape(-1, H, D)[sl, h].double().numpy())
            acc[n][1].append(ref[n][:, 0])
        for n in ("dalpha", "dmu", "deta", "dbeta"):
            acc[n][0].append(got[n].reshape(-1, H)[sl, h].double().numpy())
            acc[n][1].append(ref[n][:, 0])
        for n in ("dS0", "dM0"):
            acc[n][0].append(got[n][s, h].double().numpy())
            acc[n][1].append(ref[n][0, 0])
    errs = {}
    for n, (a, b) in acc.items():
        a, b = np.concatenate([np.ravel(t) for t in a]), np.concatenate([np.ravel(t) for t in b])
        den = np.linalg.norm(b)
        errs[n] = float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))
    print("gradient rel L2 (%s):" % x["dtype"],
          " ".join("%s %.2e" % (n, e) for n, e in errs.items()))
    for n, e in errs.items():
        assert np.isfinite(e), (n, e)
        assert e <= tol, "%s rel L2 %.3e > %.1e (%s)" % (n, e, tol, errs)
    return errs


@pytest.mark.parametrize("dtype,D", [("fp32", 64), ("fp32", 128), ("bf16", 128), ("bf16", 64)])
@pytest.mark.parametrize("T", [64, 130])
def test_small_equal_lengths(dtype, D, T):
    w = W.Workload("bwd_small", dtype=dtype, state="randn", seed=51)
    x = W.make_prefill(w, B=2, T=T, H=2, D=D, with_beta=True)
    do, dS, dM = _adjoints(x, 52)
    _compare(x, _gpu_grads(x, do, dS, dM), do, dS, dM, chains(x))


def test_tiny_fp32_workload():
    x = W.make_prefill(W.TINY_FP32)
    do, dS, dM = _adjoints(x, 53)
    _compare(x, _gpu_grads(x, do, dS, dM), do, dS, dM, chains(x))


def test_beta_absent_and_no_state_adjoints():
    w = W.Workload("bwd_nobeta", dtype="fp32", state="zero", seed=54)
    x = W.make_prefill(w, B=1, T=200, H=2, D=128)
    do, _, _ = _adjoints(x, 55, with_state_adjoints=False)
    _compare(x, _gpu_grads(x, do, None, None), do, None, None, chains(x))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_mu_zero_and_beta_zero(dtype):
    w = W.Workload("bwd_edge", dtype=dtype, state="randn", seed=56)
    x = W.make_prefill(w, B=1, T=150, H=2, D=128, with_beta=True)
    x["mu"][:, ::5] = 0.0
    x["mu"][:, 70:80] = 0.0
    x["beta"][:, 3::7] = 0.0
    x["alpha"][:, 100:110] = 1.0
    do, dS, dM = _adjoints(x, 57)
    _compare(x, _gpu_grads(x, do, dS, dM), do, dS, dM, chains(x))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_packed_with_empty_sequences(dtype):
    w = W.Workload("bwd_var", dtype=dtype, state="randn", seed=58)
    x = W.make_prefill(w, H=2, D=128, lengths=[1, 64, 0, 65, 130, 7, 0], with_beta=True)
    do, dS, dM = _adjoints(x, 59)
    got = _gpu_grads(x, do, dS, dM)
    _compare(x, got, do, dS, dM, chains(x))
    # empty sequences pass the state adjoints through unchanged
    for s in (2, 6):
        assert torch.equal(got["dS0"][s], dS[s]) and torch.equal(got["dM0"][s], dM[s])


def _sample(x, n, seed):
    ch = chains(x)
    g = torch.Generator().manual_seed(seed)
    idx = torch.randperm(len(ch), generator=g)[:n].tolist()
    return [ch[i] for i in sorted(idx)]


@pytest.mark.parametrize("w", [W.PREFILL_400M, W.PREFILL_1P3B_LONG, W.VARLEN_PACKED],
                         ids=lambda w: w.name)
def test_full_size_sampled(w):
    x = W.make_prefill(w)
    do, dS, dM = _adjoints(x, 60)
    got = _gpu_grads(x, do, dS, dM)
    for n in ("dq", "dk", "dv", "dalpha", "dmu", "deta"):
        assert torch.isfinite(got[n].float()).all(), n
    _compare(x, got, do, dS, dM, _sample(x, 2, 61))


def test_deterministic():
    w = W.Workload("bwd_det", dtype="bf16", state="randn", seed=62)
    x = W.make_prefill(w, B=2, T=300, H=2, D=128, with_beta=True)
    do, dS, dM = _adjoints(x, 63)
    a = _gpu_grads(x, do, dS, dM)
    b = _gpu_grads(x, do, dS, dM)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_many_chains_dual_slice_forward():
    """Enough (sequence, head) chains that the forward's state pass carries
    both 64-column slices of a head per CTA: the gradient from the entry
    states that kernel saved."""
    w = W.Workload("bwd_dual", dtype="bf16", state="randn", seed=64)
    x = W.make_prefill(w, B=40, T=130, H=2, D=128, with_beta=True)
    do, dS, dM = _adjoints(x, 65)
    _compare(x, _gpu_grads(x, do, dS, dM), do, dS, dM, chains(x)[::9])


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_no_tokens_passes_state_adjoints_through(dtype):
    """Sequences without tokens: nothing depends on the inputs, and the
    initial states' gradients are the final states' adjoints unchanged."""
    w = W.Workload("bwd_empty", dtype=dtype, state="randn", seed=66)
    x = W.make_prefill(w, H=2, D=128, lengths=[0, 0, 0])
    do, dS, dM = _adjoints(x, 67)
    got = _gpu_grads(x, do, dS, dM)
    assert got["dq"].numel() == 0
    assert torch.equal(got["dS0"], dS) and torch.equal(got["dM0"], dM)


@pytest.mark.parametrize("lengths,B,T,H", [
    (None, 3, 150, 2),                          # equal lengths, ragged last chunk
    ([1, 64, 0, 65, 130, 7, 0], 1, None, 2),    # packed with empty members
    (None, 40, 130, 2),                         # both slices of a head per state CTA
])
def test_forward_workspace_reuse_is_bit_identical(lengths, B, T, H):
    """The gradient that takes T and A_O T from the state-saving forward's
    workspace (its prep kernel skipped) equals, bit for bit, the gradient
    that recomputes them."""
    import momentum_delta_rule_gb300 as mdn
    w = W.Workload("bwd_reuse", dtype="bf16", state="randn", seed=61)
    if lengths is None:
        x = W.make_prefill(w, B=B, T=T, H=H, D=128, with_beta=True)
    else:
        x = W.make_prefill(w, H=H, D=128, lengths=lengths, with_beta=True)
    do, dS, dM = _adjoints(x, 62)
    d = to_dev(x)
    n_seq = x["n_seq"]
    fws = torch.empty(max(256, mdn.workspace_size(n_seq, d["q"].shape[0] * d["q"].shape[1], H, 128,
                                                  d["q"].dtype)), dtype=torch.uint8, device="cuda")
    _, _, _, Sc, Mc = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                                    d["beta"], d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"],
                                    workspace=fws, return_chunk_states=True)
    args = (d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], Sc, Mc, do.cuda())
    kw = dict(beta=d["beta"], dS_T=dS.cuda(), dM_T=dM.cuda(), cu_seqlens=d["cu_seqlens"])
    g0 = mdn.chunk_bwd(*args, **kw)
    g1 = mdn.chunk_bwd(*args, fwd_workspace=fws, **kw)
    torch.cuda.synchronize()
    assert mdn.device_status() == mdn.MDN_OK
    for n in g0:
        if g0[n] is None:
            assert g1[n] is None
            continue
        assert torch.equal(g0[n], g1[n]), n
