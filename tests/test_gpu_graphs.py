"""The library's calls inside CUDA graphs: a prefill (packed sequences, so
the chunk-offset, prep and state-pass launches, the last a programmatic
dependent launch, are all captured) and a run of decode steps are captured
once, replayed on new inputs written into the captured buffers, and must
match direct calls bit for bit."""
import pytest
import torch

import workloads as W
from tests._helpers import gpu_chunk_fwd, to_dev

pytestmark = pytest.mark.gpu


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):      # warm-up outside the capture
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_chunk_fwd_graph_replay(dtype, D):
    import momentum_delta_rule_gb300 as mdn
    lengths = [100, 0, 257, 64, 1]
    base = W.Workload("graph_prefill", dtype=dtype, state="randn", seed=61)
    x1 = W.make_prefill(base, H=4, D=D, lengths=lengths, with_beta=True)
    x2 = W.make_prefill(W.Workload("graph_prefill2", dtype=dtype, state="randn", seed=62),
                        H=4, D=D, lengths=lengths, with_beta=True)
    d = to_dev(x1)
    names = ["q", "k", "v", "alpha", "mu", "eta", "beta", "S0", "M0"]
    n_seq = d["n_seq"]
    o = torch.empty_like(d["v"])
    S_T = torch.empty((n_seq, 4, D, D), device="cuda")
    M_T = torch.empty_like(S_T)
    ws = torch.empty(mdn.workspace_size(n_seq, d["q"].shape[1], 4, D, d["q"].dtype),
                     dtype=torch.uint8, device="cuda")

    def run():
        mdn.chunk_fwd(*(d[n] for n in names), cu_seqlens=d["cu_seqlens"], o=o, S_T=S_T,
                      M_T=M_T, workspace=ws)

    g = _capture(run)
    for n in names:                    # new inputs into the captured buffers
        d[n].copy_(x2[n].to("cuda"))
    g.replay()
    torch.cuda.synchronize()
    ref = gpu_chunk_fwd(x2)
    assert torch.equal(o, ref[0]) and torch.equal(S_T, ref[1]) and torch.equal(M_T, ref[2])


def test_chunk_fwd_time_segments_graph_replay():
    """A long equal-length prefill that runs in time segments (each later
    segment's prep a programmatic dependent of the previous segment's state
    pass) captured and replayed on new inputs."""
    import momentum_delta_rule_gb300 as mdn
    B, T, H, D = 1, 8256, 2, 128
    x1 = W.make_prefill(W.Workload("graph_seg", dtype="bf16", state="randn", seed=63),
                        B=B, T=T, H=H, D=D)
    x2 = W.make_prefill(W.Workload("graph_seg2", dtype="bf16", state="randn", seed=64),
                        B=B, T=T, H=H, D=D)
    d = to_dev(x1)
    names = ["q", "k", "v", "alpha", "mu", "eta", "S0", "M0"]
    o = torch.empty_like(d["v"])
    S_T = torch.empty((B, H, D, D), device="cuda")
    M_T = torch.empty_like(S_T)
    ws = torch.empty(mdn.workspace_size(B, B * T, H, D, d["q"].dtype), dtype=torch.uint8,
                     device="cuda")

    def run():
        mdn.chunk_fwd(*(d[n] for n in names[:6]), None, d["S0"], d["M0"], o=o, S_T=S_T,
                      M_T=M_T, workspace=ws)

    g = _capture(run)
    for n in names:
        d[n].copy_(x2[n].to("cuda"))
    g.replay()
    torch.cuda.synchronize()
    ref = gpu_chunk_fwd(x2)
    assert torch.equal(o, ref[0]) and torch.equal(S_T, ref[1]) and torch.equal(M_T, ref[2])


def test_decode_steps_graph_replay():
    import momentum_delta_rule_gb300 as mdn
    w = W.Workload("graph_decode", B=8, T=1, H=4, D=128, dtype="bf16", state="randn",
                   decode_steps=6, seed=63)
    S0, M0 = W.make_decode_state(w, device="cuda")
    xs = W.make_decode_steps(w, 6, device="cuda")
    S, M = S0.clone(), M0.clone()
    o = torch.empty_like(xs["v"][0])
    outs = torch.empty((3,) + tuple(o.shape), dtype=o.dtype, device="cuda")
    step_in = {n: xs[n][0].clone() for n in ("q", "k", "v", "alpha", "mu", "eta")}

    def run():                         # three steps on the same step buffers
        for t in range(3):
            mdn.decode_step(step_in["q"], step_in["k"], step_in["v"], step_in["alpha"],
                            step_in["mu"], step_in["eta"], S, M, o=o)
            outs[t].copy_(o)

    g = _capture(run)                  # the warm-up advanced S, M: start again
    S.copy_(S0)
    M.copy_(M0)
    for n in step_in:
        step_in[n].copy_(xs[n][3])
    g.replay()
    torch.cuda.synchronize()
    S2, M2 = S0.clone(), M0.clone()
    ref = []
    for t in range(3):
        ref.append(mdn.decode_step(xs["q"][3], xs["k"][3], xs["v"][3], xs["alpha"][3],
                                   xs["mu"][3], xs["eta"][3], S2, M2).clone())
    torch.cuda.synchronize()
    for t in range(3):
        assert torch.equal(outs[t], ref[t])
    assert torch.equal(S, S2) and torch.equal(M, M2)


def test_chunk_bwd_graph_replay():
    """The gradient pass (packed sequences, bf16: the offsets, the forward's
    prep, the coefficient, chain, chunk and gate kernels) captured once and
    replayed on new inputs and saved states written into the captured
    buffers: bit for bit the direct call's gradients."""
    import momentum_delta_rule_gb300 as mdn
    lengths = [100, 0, 257, 64, 1]
    xs = [W.make_prefill(W.Workload("graph_bwd%d" % i, dtype="bf16", state="randn", seed=70 + i),
                         H=2, D=128, lengths=lengths, with_beta=True) for i in range(2)]

    def inputs(x):
        d = to_dev(x)
        _, _, _, Sc, Mc = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                                        d["beta"], d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"],
                                        return_chunk_states=True)
        g = torch.Generator(device="cuda").manual_seed(80)
        d["do"] = torch.randn(d["v"].shape, generator=g, device="cuda").to(d["v"].dtype)
        d["dS"] = torch.randn(d["S0"].shape, generator=g, device="cuda") * 0.1
        d["dM"] = torch.randn(d["M0"].shape, generator=g, device="cuda") * 0.1
        d["Sc"], d["Mc"] = Sc, Mc
        return d

    d, d2 = inputs(xs[0]), inputs(xs[1])
    need = mdn.chunk_bwd_workspace_size(d["n_seq"], d["q"].shape[1], 2, 128, d["q"].dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = {}

    def call(e):
        return mdn.chunk_bwd(e["q"], e["k"], e["v"], e["alpha"], e["mu"], e["eta"], e["Sc"],
                             e["Mc"], e["do"], beta=e["beta"], dS_T=e["dS"], dM_T=e["dM"],
                             cu_seqlens=e["cu_seqlens"], workspace=ws)

    def run():
        out["g"] = call(d)

    g = _capture(run)
    for n in ("q", "k", "v", "alpha", "mu", "eta", "beta", "Sc", "Mc", "do", "dS", "dM"):
        d[n].copy_(d2[n])
    g.replay()
    torch.cuda.synchronize()
    ref = call(d2)
    torch.cuda.synchronize()
    for n, t in out["g"].items():
        assert torch.equal(t, ref[n]), n
    assert mdn.device_status() == mdn.MDN_OK
