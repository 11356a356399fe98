"""GPU parity of the 64-column state slices of the tensor-core state pass,
which run once there are more (sequence, head) chains than 32-column slices
fit on the GPU in one wave (>= 39 chains on 152 SMs).

Every case here has at least 48 chains; the edge cases of the narrow-slice
tests are repeated: ragged and one-token chunks, mu = 0 and beta = 0
entries, alpha = 1 runs, nonzero initial states, packed sequences with empty
members, and the per-token residual output.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import recurrence
from tests._helpers import TOL, chains, compare, gpu_chunk_fwd, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
def test_wide_ragged(T):
    w = W.Workload("wide", dtype="bf16", state="randn", seed=41)
    x = W.make_prefill(w, B=3, T=T, H=16, D=128, with_beta=True)
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_wide_gate_edges():
    w = W.Workload("wide_edge", dtype="bf16", state="randn", seed=42)
    x = W.make_prefill(w, B=3, T=200, H=16, D=128, with_beta=True)
    x["mu"][:, ::5] = 0.0
    x["mu"][:, 70:80] = 0.0
    x["beta"][:, 3::7] = 0.0
    x["alpha"][:, 100:110] = 1.0
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_wide_varlen_with_empty_sequences():
    x = W.make_prefill(W.VARLEN_PACKED, H=8, lengths=[1, 64, 0, 65, 130, 7, 0, 200])
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_wide_residuals_and_bitwise_repeat():
    import momentum_delta_rule_gb300 as mdn
    w = W.Workload("wide_vres", dtype="bf16", state="randn", seed=43)
    x = W.make_prefill(w, B=3, T=150, H=16, D=128, with_beta=True)
    d = to_dev(x)
    o, S_T, M_T, vres = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"],
                                      d["eta"], d["beta"], d["S0"], d["M0"],
                                      return_vres=True)
    o2, S2, M2 = gpu_chunk_fwd(x)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(S_T, S2) and torch.equal(M_T, M2)
    sel = chains(x)[::7]
    compare(x, (o, S_T, M_T), sel)
    D, H = x["D"], x["H"]
    flat = vres.reshape(-1, H, D).double().cpu().numpy()
    got, want = [], []
    for (s, h, sl) in sel:
        L = sl.stop - sl.start
        ref = recurrence.forward(
            x["q"].reshape(-1, H, D)[sl, h][:, None], x["k"].reshape(-1, H, D)[sl, h][:, None],
            x["v"].reshape(-1, H, D)[sl, h][:, None], x["alpha"].reshape(-1, H)[sl, h][:, None],
            x["mu"].reshape(-1, H)[sl, h][:, None], x["eta"].reshape(-1, H)[sl, h][:, None],
            x["beta"].reshape(-1, H)[sl, h][:, None], x["S0"][s, h][None, None],
            x["M0"][s, h][None, None], cu_seqlens=[0, L], return_vres=True)
        got.append(flat[sl, h])
        want.append(ref[3][:, 0])
    got, want = np.concatenate(got), np.concatenate(want)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= TOL["bf16"]
