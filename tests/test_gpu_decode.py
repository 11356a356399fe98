"""GPU parity of mdn_decode_step (through the C ABI) against the fp64 oracle."""
import pytest
import torch

import workloads as W
from oracle import recurrence

pytestmark = pytest.mark.gpu


def _run(w, steps, N, H, D, sample=None, with_beta=False):
    import momentum_delta_rule_gb300 as mdn
    S, M = W.make_decode_state(w, N=N, H=H, D=D)
    xs = W.make_decode_steps(w, steps, N=N, H=H, D=D, with_beta=with_beta)
    Sd, Md = S.cuda(), M.cuda()
    xd = {k: (v.cuda() if v is not None else None) for k, v in xs.items()}
    outs = []
    for t in range(steps):
        o = mdn.decode_step(xd["q"][t], xd["k"][t], xd["v"][t], xd["alpha"][t],
                            xd["mu"][t], xd["eta"][t], Sd, Md,
                            beta=None if xd["beta"] is None else xd["beta"][t])
        outs.append(o)
    torch.cuda.synchronize()
    o_gpu = torch.stack(outs).float().cpu()           # [steps, N, H, D]
    # oracle on the selected (n, h) chains, all steps
    sel = sample if sample is not None else [(n, h) for n in range(N) for h in range(H)]
    ns = torch.tensor([s[0] for s in sel])
    hs = torch.tensor([s[1] for s in sel])
    So = S[ns, hs].double().numpy()[:, None]           # [n_sel, 1, D, D]
    Mo = M[ns, hs].double().numpy()[:, None]
    o_ref = []
    for t in range(steps):
        pick = lambda a: a[t][ns, hs][:, None]
        o, So, Mo = recurrence.decode_step(
            pick(xs["q"]), pick(xs["k"]), pick(xs["v"]), pick(xs["alpha"]),
            pick(xs["mu"]), pick(xs["eta"]), So, Mo,
            beta=None if xs["beta"] is None else pick(xs["beta"]))
        o_ref.append(o[:, 0])
    o_ref = torch.from_numpy(__import__("numpy").stack(o_ref))   # [steps, n_sel, D]
    o_sel = o_gpu[:, ns, hs]
    tol = 1e-4 if w.dtype == "fp32" else 2e-2
    e_o = W.rel_l2(o_sel, o_ref)
    e_S = W.rel_l2(Sd.cpu()[ns, hs], torch.from_numpy(So[:, 0]))
    e_M = W.rel_l2(Md.cpu()[ns, hs], torch.from_numpy(Mo[:, 0]))
    assert e_o <= tol and e_S <= tol and e_M <= tol, (e_o, e_S, e_M)
    return e_o, e_S, e_M


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 128), ("fp32", 64), ("bf16", 64)])
def test_decode_small(dtype, D):
    w = W.Workload("dec_small", B=3, H=2, D=D, dtype=dtype, seed=21)
    _run(w, 20, 3, 2, D, with_beta=True)


def test_decode_full_size_sampled():
    """The 256 x 16 x 128 workload for all 1000 steps; 24 sampled chains."""
    w = W.DECODE
    g = torch.Generator().manual_seed(5)
    sel = sorted({(int(n), int(h)) for n, h in zip(
        torch.randint(0, w.B, (24,), generator=g), torch.randint(0, w.H, (24,), generator=g))})
    _run(w, w.decode_steps, w.B, w.H, w.D, sample=sel)
