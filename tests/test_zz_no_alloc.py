"""The allocation-free prefill entry point, mdn_chunk_fwd_static_ws.

Some callers cannot allocate device memory where they run the prefill (a
server that reserves all device memory at start and forbids allocation later,
because cudaMalloc may synchronise the device and take unbounded time, or
plugin code without access to its host's allocator).  For them the library
keeps a fixed 32 MiB scratch array of its own.  This test calls that entry
point directly through the C ABI three times in a row on different inputs
(a larger problem, a smaller one, the larger one again, so a call that read
the previous call's leftover scratch would show) and checks each result
against the regular entry point (caller-provided workspace).  Both run the
same deterministic kernels on the same inputs, so the outputs must be
identical bit for bit.  It lives in a file of its own that pytest collects
last.
"""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_call(L, x, o, S_T, M_T, stream):
    B, T, H, D = x["q"].shape
    return L.mdn_chunk_fwd_static_ws(
        _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["alpha"]), _p(x["mu"]),
        _p(x["eta"]), _p(x["beta"]), _p(x["S0"]), _p(x["M0"]), _p(o), _p(S_T),
        _p(M_T), _p(x["cu_seqlens"]), x["n_seq"], B, T, H, D, D, 1, 64,
        ctypes.c_void_p(stream.cuda_stream))


def test_static_workspace_matches_regular_entry_point():
    import momentum_delta_rule_gb300 as mdn
    L = mdn.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    large = W.make_prefill(W.Workload("noalloc_a", dtype="bf16", state="randn", seed=31),
                           B=2, T=300, H=4, D=128, with_beta=True)
    small = W.make_prefill(W.VARLEN_PACKED, H=4, lengths=[100, 0, 257, 64, 1], seed=32)
    for x in (large, small, large):       # three calls in a row
        x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        o_ref, S_ref, M_ref = mdn.chunk_fwd(
            x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
            x["S0"], x["M0"], cu_seqlens=x["cu_seqlens"])
        o = torch.empty_like(o_ref)
        S_T = torch.empty_like(S_ref)
        M_T = torch.empty_like(M_ref)
        st = _static_call(L, x, o, S_T, M_T, stream)
        assert st == 0, mdn.status_string(st)
        torch.cuda.synchronize()
        assert mdn.device_status() == 0
        assert torch.equal(o, o_ref)
        assert torch.equal(S_T, S_ref) and torch.equal(M_T, M_ref)


def test_static_workspace_rejects_oversized_problem():
    import momentum_delta_rule_gb300 as mdn
    L = mdn.lib()
    dev = torch.device("cuda", 0)
    B, T, H, D = 8, 2048, 8, 128          # needs far more than 32 MiB of scratch
    assert mdn.workspace_size(B, B * T, H, D, 1) > (32 << 20)
    q = torch.zeros(B, T, H, D, dtype=torch.bfloat16, device=dev)
    g = torch.zeros(B, T, H, device=dev)
    x = dict(q=q, k=q, v=q, alpha=g, mu=g, eta=g, beta=None, S0=None, M0=None,
             cu_seqlens=None, n_seq=B)
    o = torch.empty_like(q)
    st = _static_call(L, x, o, None, None, torch.cuda.current_stream(dev))
    assert st == mdn.MDN_ERR_UNSUPPORTED
