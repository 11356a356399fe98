"""GPU parity of mdn_chunk_fwd (through the C ABI) against the fp64 oracle.

Small cases compare every output; the full-size workloads run exactly as the
bench launches them and compare sampled independent (sequence, head) chains,
each against a full oracle run of that chain.
"""
import pytest
import torch

import workloads as W
from tests._helpers import TOL, chains, compare, gpu_chunk_fwd

pytestmark = pytest.mark.gpu


def _sample(x, n, seed=0):
    ch = chains(x)
    g = torch.Generator().manual_seed(seed)
    idx = torch.randperm(len(ch), generator=g)[:n].tolist()
    return [ch[i] for i in sorted(idx)]


def test_tiny_fp32_full_parity():
    x = W.make_prefill(W.TINY_FP32)
    out = gpu_chunk_fwd(x)
    errs = compare(x, out, chains(x))
    assert errs["o"] <= TOL["fp32"]


def test_tiny_fp32_with_beta():
    x = W.make_prefill(W.TINY_FP32, with_beta=True)
    compare(x, gpu_chunk_fwd(x), chains(x))


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 128), ("bf16", 64)])
def test_small_ragged(T, dtype, D):
    w = W.Workload("small", dtype=dtype, state="randn", seed=11)
    x = W.make_prefill(w, B=2, T=T, H=2, D=D, with_beta=True)
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_varlen_small_with_empty_sequences():
    x = W.make_prefill(W.VARLEN_PACKED, H=2, lengths=[1, 64, 0, 65, 130, 7, 0])
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_mu_zero_and_beta_zero():
    w = W.Workload("edge", dtype="bf16", state="randn", seed=12)
    x = W.make_prefill(w, B=1, T=150, H=2, D=128, with_beta=True)
    x["mu"][:, ::5] = 0.0
    x["mu"][:, 70:80] = 0.0
    x["beta"][:, 3::7] = 0.0
    x["alpha"][:, 100:110] = 1.0
    compare(x, gpu_chunk_fwd(x), chains(x))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 128)])
def test_gate_extremes(dtype, D):
    """Gates at the ends of their ranges: alpha down to 1e-4 (the chunk's
    alpha product underflows fp32 well inside a chunk), mu = 1 exactly over
    whole chunks (momentum never decays), mu = 0 runs, eta up to 2, beta up
    to 3, and tokens with alpha = 1 and eta = 0 (no write at all)."""
    w = W.Workload("gate_edges", dtype=dtype, state="randn", seed=15)
    x = W.make_prefill(w, B=2, T=260, H=2, D=D, with_beta=True)
    g = torch.Generator().manual_seed(16)
    x["alpha"][:, 0:40] = 10.0 ** (-4.0 * torch.rand(x["alpha"][:, 0:40].shape, generator=g))
    x["mu"][:, 64:192] = 1.0
    x["mu"][:, 200:210] = 0.0
    x["eta"][:, 120:180] = 2.0 * torch.rand(x["eta"][:, 120:180].shape, generator=g)
    x["beta"][:, 150:230] = 3.0 * torch.rand(x["beta"][:, 150:230].shape, generator=g)
    x["alpha"][:, 240:250] = 1.0
    x["eta"][:, 240:250] = 0.0
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_state_alias_and_optional_states():
    import momentum_delta_rule_gb300 as mdn
    w = W.Workload("alias", dtype="bf16", state="randn", seed=13)
    x = W.make_prefill(w, B=2, T=100, H=2, D=128)
    ref = gpu_chunk_fwd(x)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    S, M = d["S0"].clone(), d["M0"].clone()
    o, S_T, M_T = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"],
                                d["eta"], None, S, M, S_T=S, M_T=M)
    torch.cuda.synchronize()
    assert torch.equal(o, ref[0]) and torch.equal(S, ref[1]) and torch.equal(M, ref[2])
    o2, S2, M2 = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"],
                               d["eta"], None, d["S0"], d["M0"],
                               output_final_state=False)
    torch.cuda.synchronize()
    assert S2 is None and M2 is None and torch.equal(o2, ref[0])


def test_deterministic():
    x = W.make_prefill(W.PREFILL_400M, B=2, T=300, H=4)
    a = gpu_chunk_fwd(x)
    b = gpu_chunk_fwd(x)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_split_sequence_state_passing():
    """fwd(x) equals fwd(second half) started from fwd(first half)'s states."""
    w = W.Workload("split", dtype="bf16", state="randn", seed=14)
    x = W.make_prefill(w, B=1, T=256, H=2, D=128)
    full = gpu_chunk_fwd(x)
    first = dict(x)
    for n in ("q", "k", "v", "alpha", "mu", "eta"):
        first[n] = x[n][:, :128].contiguous()
    first["T"] = 128
    o1, S1, M1 = gpu_chunk_fwd(first)
    second = dict(x)
    for n in ("q", "k", "v", "alpha", "mu", "eta"):
        second[n] = x[n][:, 128:].contiguous()
    second["S0"], second["M0"] = S1.cpu(), M1.cpu()
    o2, S2, M2 = gpu_chunk_fwd(second)
    rel = lambda a, b: ((a.float() - b.float()).norm() / b.float().norm()).item()
    assert rel(torch.cat([o1, o2], 1), full[0]) < 1e-2
    assert rel(S2, full[1]) < 1e-3 and rel(M2, full[2]) < 1e-3


@pytest.mark.parametrize("D,B,T,H", [(128, 1, 9000, 3), (64, 1, 8256, 3), (128, 1, 8256, 24),
                                     (128, 2, 8200, 4)])
def test_time_segments_bit_identical(D, B, T, H):
    """Long equal-length sequences whose state pass runs narrow slices are
    walked in time segments, the prep of the next segment beside the state
    pass of the current one, each segment starting from the states the
    previous one left in S_T, M_T.  The segments' kernels do the same
    arithmetic as one pass over whole sequences, which runs when no final
    states are asked for: the outputs match it bit for bit, also with the
    final states written over the initial ones (S_T aliasing S0); one chain
    against the oracle."""
    import momentum_delta_rule_gb300 as mdn
    w = W.Workload("segments", dtype="bf16", state="randn", seed=19)
    x = W.make_prefill(w, B=B, T=T, H=H, D=D, with_beta=True)
    # four segments (16, 32, 64 and the rest), two kernels each, on 16- or
    # (24 heads of 128) 32-column slices; one pass without final states
    assert mdn.chunk_fwd_kernel_count(B, B, T, H, D, torch.bfloat16, False) == 8
    assert mdn.chunk_fwd_kernel_count(B, B, T, H, D, torch.bfloat16, False, False) == 2
    seg = gpu_chunk_fwd(x)
    whole = gpu_chunk_fwd(x, output_final_state=False)
    assert whole[1] is None
    assert torch.equal(seg[0], whole[0])
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    S, M = d["S0"].clone(), d["M0"].clone()
    o, S_T, M_T = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                                d["beta"], S, M, S_T=S, M_T=M)
    torch.cuda.synchronize()
    assert torch.equal(o, seg[0]) and torch.equal(S, seg[1]) and torch.equal(M, seg[2])
    compare(x, seg, chains(x)[:1] + chains(x)[-1:])


# ---------------------------------------------------------------- full size

def test_prefill_400m_full_size_sampled():
    x = W.make_prefill(W.PREFILL_400M)
    out = gpu_chunk_fwd(x)
    compare(x, out, _sample(x, 4))


def test_prefill_1p3b_long_full_size_sampled():
    x = W.make_prefill(W.PREFILL_1P3B_LONG)
    out = gpu_chunk_fwd(x)
    compare(x, out, _sample(x, 2))


def test_varlen_packed_full_size_sampled():
    x = W.make_prefill(W.VARLEN_PACKED)
    out = gpu_chunk_fwd(x)
    ch = chains(x)
    shortest = min(ch, key=lambda c: c[2].stop - c[2].start)
    compare(x, out, _sample(x, 4) + [shortest])


def test_fp32_many_chains_two_waves():
    """fp32 inputs at d = 128 with more chains than 32-column CTAs fit in one
    wave (>= 39 chains on 152 SMs): the split-operand state pass keeps
    32-column slices and runs two waves; ragged chunks and mu = 0 entries."""
    w = W.Workload("fp32_wide", dtype="fp32", state="randn", seed=18)
    x = W.make_prefill(w, B=3, T=130, H=16, D=128, with_beta=True)
    x["mu"][:, ::7] = 0.0
    compare(x, gpu_chunk_fwd(x), chains(x)[::6])


def test_very_long_sequence_sampled():
    """One sequence of 131072 tokens: a chain of 2048 chunks, eight times the
    longest benchmark sequence; one head compared in full against the
    oracle, so error growth along the chain would show."""
    w = W.Workload("very_long", dtype="bf16", state="randn", seed=17)
    x = W.make_prefill(w, B=1, T=131072, H=2, D=128)
    out = gpu_chunk_fwd(x)
    compare(x, out, chains(x)[:1])


def test_path_selection():
    """Every input runs on the tensor-core path: bf16 directly, fp32 as hi /
    lo bf16 parts, head size 64 and 128 alike."""
    import momentum_delta_rule_gb300 as mdn
    for dtype, D in (("bf16", 128), ("fp32", 128), ("bf16", 64), ("fp32", 64)):
        w = W.Workload("path", dtype=dtype, state="zero", seed=15)
        x = W.make_prefill(w, B=1, T=70, H=1, D=D)
        info = {}
        gpu_chunk_fwd(x, info=info)
        assert info["path"] == mdn.MDN_PATH_TENSOR_CORE, (dtype, D, info)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 128), ("bf16", 64), ("fp32", 64)])
@pytest.mark.parametrize("B,H", [(2, 2), (5, 5), (5, 10), (7, 11)])
def test_slice_widths(B, H, dtype, D):
    """The tensor-core state pass picks 16-, 32- or 64-column state slices by
    the number of (sequence, head) chains (4, 25 and 50 chains here select
    each width on a 152-SM GPU at head size 128; fp32 there stops at 32), and
    beyond one wave of 64-column slices (77 chains, bf16, head size 128) both
    slices of a head in one CTA; every form must match the oracle."""
    w = W.Workload("widths", dtype=dtype, state="randn", seed=16)
    x = W.make_prefill(w, B=B, T=130, H=H, D=D, with_beta=True)
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_fp32_prefill_400m_shapes_sampled():
    """fp32 inputs at the 400M-model shapes (B8 H8 T2048 d128) on the
    tensor cores with split operands: sampled chains within the fp32
    tolerance."""
    w = W.Workload("fp32_400m", dtype="fp32", state="zero", seed=1)
    x = W.make_prefill(w, B=8, T=2048, H=8, D=128)
    compare(x, gpu_chunk_fwd(x), _sample(x, 3, seed=5))


def test_fp32_packed_with_empty_sequences():
    w = W.Workload("fp32_var", dtype="fp32", state="randn", seed=18)
    x = W.make_prefill(w, H=2, D=64, lengths=[1, 64, 0, 65, 130, 7, 0], with_beta=True)
    compare(x, gpu_chunk_fwd(x), chains(x))


def test_dual_slices_packed_with_empty_sequences():
    """More (sequence, head) chains than one wave of 64-column slices holds
    (bf16, d = 128): one CTA carries both slices of a head, their steps
    interleaved.  Packed sequences of every ragged length, empty members,
    initial states, beta and mu = 0 entries."""
    lengths = [1, 63, 64, 65, 0, 130, 7, 200, 0, 129] * 5
    w = W.Workload("dual", dtype="bf16", state="randn", seed=19)
    x = W.make_prefill(w, H=4, D=128, lengths=lengths, with_beta=True)
    x["mu"][:, ::9] = 0.0
    out = gpu_chunk_fwd(x)
    compare(x, out, chains(x)[::7])
