"""GPU parity of the token-mixer block (mdn_block_fwd, through the C ABI)
against the fp64 block oracle (oracle/block.py), at the forward's
tolerances (relative L2 of y, S_T and M_T: 1e-4 for fp32, 2e-2 for bf16).
Weights are seeded random draws (the block needs no trained weights to be
checked); inputs are rounded to the run's dtype before the oracle sees them.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import block
from tests._helpers import TOL

pytestmark = pytest.mark.gpu

GP = dict(a=1.0, b=0.0, s=1.0, tau=8.0, log_mu_min=-2.0, comba_d=0.1)


def _case(dtype, H, d, d_model, lengths=None, B=1, T=0, seed=0, state=False):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    if lengths is not None:
        T_total = sum(lengths)
        cu = torch.tensor(np.cumsum([0] + list(lengths)), dtype=torch.int32)
        B_, T_, n_seq = 1, T_total, len(lengths)
    else:
        T_total, cu, B_, T_, n_seq = B * T, None, B, T, B
    n_in = 4 * H * d + 4 * H
    x = torch.randn((B_, T_, d_model), generator=g).to(tdt)
    W_in = (torch.randn((d_model, n_in), generator=g) / d_model ** 0.5).to(tdt)
    conv_w = torch.randn((3 * H * d, 4), generator=g) * 0.5
    rms_w = 1.0 + 0.1 * torch.randn((d,), generator=g)
    W_o = (torch.randn((H * d, d_model), generator=g) / (H * d) ** 0.5).to(tdt)
    S0 = M0 = None
    if state:
        S0 = torch.randn((n_seq, H, d, d), generator=g) * 0.01
        M0 = torch.randn((n_seq, H, d, d), generator=g) * 0.01
    return dict(x=x, W_in=W_in, conv_w=conv_w, rms_w=rms_w, W_o=W_o, cu=cu, S0=S0, M0=M0,
                H=H, d=d, dtype=dtype, n_seq=n_seq)


def _check(c):
    import momentum_delta_rule_gb300 as mdn
    dev = lambda t: None if t is None else t.cuda()
    y, S_T, M_T = mdn.block_fwd(dev(c["x"]), dev(c["W_in"]), dev(c["conv_w"]), dev(c["rms_w"]),
                                dev(c["W_o"]), c["H"], c["d"], S0=dev(c["S0"]), M0=dev(c["M0"]),
                                cu_seqlens=dev(c["cu"]), **GP)
    torch.cuda.synchronize()
    assert mdn.device_status() == mdn.MDN_OK
    f = lambda t: None if t is None else t.double().numpy()
    x = c["x"].reshape(-1, c["x"].shape[-1])
    cu = None if c["cu"] is None else c["cu"].tolist()
    if cu is None and c["x"].shape[0] > 1:
        cu = [i * c["x"].shape[1] for i in range(c["x"].shape[0] + 1)]
    ry, rS, rM = block.block_forward(f(x), f(c["W_in"]), f(c["conv_w"]), f(c["rms_w"]),
                                     f(c["W_o"]), c["H"], c["d"], GP, S0=f(c["S0"]),
                                     M0=f(c["M0"]), cu_seqlens=cu)
    tol = TOL[c["dtype"]]
    errs = {}
    for name, got, ref in (("y", y.reshape(x.shape), ry), ("S_T", S_T, rS), ("M_T", M_T, rM)):
        g_ = got.double().cpu().numpy()
        errs[name] = float(np.linalg.norm(g_ - ref) / np.linalg.norm(ref))
    print("block rel L2 (%s):" % c["dtype"], errs)
    for name, e in errs.items():
        assert np.isfinite(e) and e <= tol, (name, e, errs)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp32", 128), ("bf16", 64), ("fp32", 64)])
def test_block_equal_lengths(dtype, d):
    _check(_case(dtype, H=2, d=d, d_model=96, B=2, T=150, seed=71, state=True))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_block_packed_with_empty_sequences(dtype):
    _check(_case(dtype, H=2, d=128, d_model=64, lengths=[3, 0, 130, 64, 1, 0, 70], seed=72))


def test_block_400m_shaped():
    # 400M-model-shaped heads (H 8, d 128), d_model = H d, two 512-token sequences
    _check(_case("bf16", H=8, d=128, d_model=1024, B=2, T=512, seed=73))
