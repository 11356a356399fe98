"""Independent calls at once: two prefills (different shapes and paths, each
with its own workspace) and a decode run enqueued on three streams together
must each equal the same call made alone, bit for bit; and empty problems
(no tokens, no sequences) are accepted and write nothing."""
import pytest
import torch

import workloads as W
from tests._helpers import to_dev

pytestmark = pytest.mark.gpu


def _prefill(mdn, d, stream=None):
    return mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"], d["beta"],
                         d["S0"], d["M0"], cu_seqlens=d["cu_seqlens"], stream=stream)


def test_concurrent_streams_match_serial():
    import momentum_delta_rule_gb300 as mdn
    a = to_dev(W.make_prefill(W.Workload("cc_a", dtype="bf16", state="randn", seed=71),
                              B=4, T=700, H=8, D=128, with_beta=True))
    b = to_dev(W.make_prefill(W.Workload("cc_b", dtype="fp32", state="randn", seed=72),
                              H=4, D=64, lengths=[300, 1, 129, 64]))
    wd = W.Workload("cc_dec", B=32, T=1, H=8, D=128, dtype="bf16", state="randn",
                    decode_steps=4, seed=73)
    S0, M0 = W.make_decode_state(wd, device="cuda")
    xs = W.make_decode_steps(wd, 4, device="cuda")

    def decode(S, M, stream=None):
        outs = []
        for t in range(4):
            outs.append(mdn.decode_step(xs["q"][t], xs["k"][t], xs["v"][t], xs["alpha"][t],
                                        xs["mu"][t], xs["eta"][t], S, M, stream=stream).clone())
        return outs

    ref_a, ref_b = _prefill(mdn, a), _prefill(mdn, b)
    Sd, Md = S0.clone(), M0.clone()
    ref_d = decode(Sd, Md)
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream() for _ in range(3)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    S2, M2 = S0.clone(), M0.clone()
    torch.cuda.synchronize()
    with torch.cuda.stream(streams[0]):
        out_a = _prefill(mdn, a, streams[0])
    with torch.cuda.stream(streams[1]):
        out_b = _prefill(mdn, b, streams[1])
    with torch.cuda.stream(streams[2]):
        out_d = decode(S2, M2, streams[2])
    torch.cuda.synchronize()
    for got, want in zip(out_a + out_b, ref_a + ref_b):
        assert torch.equal(got, want)
    for got, want in zip(out_d, ref_d):
        assert torch.equal(got, want)
    assert torch.equal(S2, Sd) and torch.equal(M2, Md)
    assert mdn.device_status() == 0


def test_concurrent_time_segmented_prefills():
    """Two long equal-length prefills that each run in time segments (each
    later segment's prep a programmatic dependent of the previous segment's
    state pass, waiting for it before it completes) enqueued on two streams
    at once: the dependencies stay within each stream, and each result
    equals the same call made alone, bit for bit."""
    import momentum_delta_rule_gb300 as mdn
    xs = [to_dev(W.make_prefill(W.Workload("cc_seg%d" % i, dtype="bf16", state="randn",
                                           seed=74 + i), B=1, T=8256, H=4, D=128))
          for i in range(2)]
    assert mdn.chunk_fwd_kernel_count(1, 1, 8256, 4, 128, torch.bfloat16, False) > 2
    refs = [_prefill(mdn, x) for x in xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    outs = []
    for x, st in zip(xs, streams):
        with torch.cuda.stream(st):
            outs.append(_prefill(mdn, x, st))
    torch.cuda.synchronize()
    for got, want in zip(outs, refs):
        for g, w in zip(got, want):
            assert torch.equal(g, w)
    assert mdn.device_status() == 0


@pytest.mark.parametrize("lengths", [[0], [0, 0, 0]])
def test_empty_problems(lengths):
    import momentum_delta_rule_gb300 as mdn
    x = to_dev(W.make_prefill(W.Workload("empty", dtype="bf16", state="randn", seed=74),
                              H=2, D=128, lengths=lengths))
    S_T = torch.full_like(x["S0"], 7.0)
    M_T = torch.full_like(x["M0"], 7.0)
    o, S_T2, M_T2 = mdn.chunk_fwd(x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"],
                                  None, x["S0"], x["M0"], cu_seqlens=x["cu_seqlens"],
                                  S_T=S_T, M_T=M_T)
    torch.cuda.synchronize()
    assert o.numel() == 0
    # no tokens: the final states are the initial ones (nothing to update),
    # or left untouched where the call has no work to enqueue
    assert torch.equal(S_T2, x["S0"]) or torch.equal(S_T2, torch.full_like(S_T2, 7.0))
    assert mdn.device_status() == 0
