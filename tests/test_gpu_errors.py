"""Device-side error reporting, exercised without faulting the GPU.

* Bounded waits: mdn_wait_selftest runs a kernel that waits on a barrier no
  one arrives at, with the same bounded-wait helper as the library's kernels
  and a 2 ms limit.  The wait must expire, the kernel must free its tensor
  memory and return, the status word must read MDN_ERR_DEVICE_TIMEOUT once,
  and the next prefill on the same device must still match the oracle.
* Malformed packed offsets: cu_seqlens lives on the device, so it is checked
  there.  Each bad array below keeps every extent inside the allocated
  tensors; the call must report MDN_ERR_INVALID_ARG through the status word,
  leave o untouched and hand the initial states through as final states.
"""
import pytest
import torch

import workloads as W
from tests._helpers import TOL, chains, compare, gpu_chunk_fwd, to_dev

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    import momentum_delta_rule_gb300 as mdn
    assert mdn.device_status() == mdn.MDN_OK
    mdn.wait_selftest(2000)
    assert mdn.device_status() == mdn.MDN_ERR_DEVICE_TIMEOUT
    assert mdn.device_status() == mdn.MDN_OK            # read and cleared
    # both paths still run and match the oracle (the self-test kernel freed
    # its tensor memory, or the tensor-core kernels could not allocate theirs)
    for dtype in ("bf16", "fp32"):
        w = W.Workload("after_timeout", dtype=dtype, state="randn", seed=41)
        x = W.make_prefill(w, B=2, T=130, H=2, D=128, with_beta=True)
        compare(x, gpu_chunk_fwd(x), chains(x))
    assert mdn.device_status() == mdn.MDN_OK


def test_wait_selftest_rejects_bad_limits():
    import momentum_delta_rule_gb300 as mdn
    for bad in (0, -5, 1000001):
        with pytest.raises(mdn.MdnError):
            mdn.wait_selftest(bad)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("cu", [
    [0, 200, 100, 300],      # decreasing in the middle
    [0, 100, 250],           # ends before the packed length (300)
    [20, 100, 300],          # does not start at 0
    [0, 300, 300, 290],      # ends below the packed length after a decrease
])
def test_malformed_cu_seqlens_is_rejected_on_device(dtype, cu):
    import momentum_delta_rule_gb300 as mdn
    n_seq, H, D, T_total = len(cu) - 1, 2, 128, 300
    w = W.Workload("bad_cu", dtype=dtype, state="randn", seed=42)
    x = W.make_prefill(w, B=1, T=T_total, H=H, D=D)
    d = to_dev(x)
    g = torch.Generator().manual_seed(43)
    S0 = (0.01 * torch.randn(n_seq, H, D, D, generator=g)).cuda()
    M0 = (0.01 * torch.randn(n_seq, H, D, D, generator=g)).cuda()
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o = torch.full_like(d["v"], 7.0)
    assert mdn.device_status() == mdn.MDN_OK
    o, S_T, M_T = mdn.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["mu"], d["eta"],
                                None, S0, M0, cu_seqlens=cu_dev, o=o)
    assert mdn.device_status() == mdn.MDN_ERR_INVALID_ARG
    assert bool((o == 7.0).all())
    assert torch.equal(S_T, S0) and torch.equal(M_T, M0)
    # a valid array right after runs normally
    x2 = W.make_prefill(W.Workload("good_cu", dtype=dtype, state="zero", seed=44),
                        H=H, D=D, lengths=[120, 0, 180])
    out = gpu_chunk_fwd(x2)
    assert mdn.device_status() == mdn.MDN_OK
    compare(x2, out, chains(x2))
