"""Host-side checks of the seeded input generator (no method arithmetic)."""
import torch

import workloads as W


def test_varlen_lengths_sum_and_range():
    lens = W.varlen_lengths(32768, W.VARLEN_PACKED.seed)
    assert sum(lens) == 32768
    assert all(128 <= x <= 4096 for x in lens[:-1])
    assert 1 <= lens[-1] <= 4096
    assert lens == W.varlen_lengths(32768, W.VARLEN_PACKED.seed)


def test_prefill_small_shapes_and_determinism():
    x = W.make_prefill(W.PREFILL_400M, B=2, T=70, H=3, D=16)
    y = W.make_prefill(W.PREFILL_400M, B=2, T=70, H=3, D=16)
    assert x["q"].shape == (2, 70, 3, 16) and x["q"].dtype == torch.bfloat16
    assert x["alpha"].shape == (2, 70, 3) and x["alpha"].dtype == torch.float32
    assert torch.equal(x["q"], y["q"]) and torch.equal(x["mu"], y["mu"])
    n = x["q"].float().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)
    assert float(x["alpha"].min()) >= float(torch.exp(torch.tensor(-0.1))) - 1e-6
    assert float(x["mu"].max()) <= 0.9 and float(x["mu"].min()) >= 0.0
    assert x["beta"] is None


def test_varlen_inputs():
    x = W.make_prefill(W.VARLEN_PACKED, H=2, D=16, lengths=[5, 0, 70])
    assert x["cu_seqlens"].tolist() == [0, 5, 5, 75]
    assert x["q"].shape == (1, 75, 2, 16) and x["n_seq"] == 3
    assert x["S0"] is None


def test_rel_l2():
    a = torch.tensor([3.0, 4.0], dtype=torch.float64)
    assert W.rel_l2(a, a) == 0.0
    assert abs(W.rel_l2(a * 1.01, a) - 0.01) < 1e-12
