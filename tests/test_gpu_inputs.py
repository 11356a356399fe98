"""GPU parity of mdn_prepare_inputs (through the C ABI) against the fp64
oracle of the gate parameterisation and the query/key preparation.

Tolerances (relative L2 per output tensor): gates 1e-5 (fp32 arithmetic with
CUDA's own tanh/exp/log1p, a few ulp each); q_hat, k_hat 1e-5 for fp32 and
4e-3 for bf16 (one rounding of unit vectors to 8 significant bits, 2^-9
relative, plus the fp32 sums)."""
import numpy as np
import pytest
import torch

from oracle import gates as G

pytestmark = pytest.mark.gpu

P = dict(a=1.3, b=0.7, s=1.5, tau=2.0, log_mu_min=-2.0)


def _rel(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)


def _inputs(T, H, D, dtype, seed, zero_rows=True):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, D, generator=g)
    k = torch.randn(T, H, D, generator=g)
    z = [torch.randn(T, H, generator=g) * 3 for _ in range(4)]
    if zero_rows and T > 2:
        k[1, 0] = 0.0                       # k row of norm zero
        q[2, 0] = 0.5 * k[2, 0]             # q - 0.5 k = 0 exactly (0.5 is binary)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return q.to(tdt), k.to(tdt), z


def _check(T, H, D, dtype, seed, comba_d=0.5, in_place=False):
    import momentum_delta_rule_gb300 as mdn
    q, k, z = _inputs(T, H, D, dtype, seed)
    qd, kd = q.cuda(), k.cuda()
    zd = [t.cuda() for t in z]
    kw = dict(q_out=qd, k_out=kd) if in_place else {}
    out = mdn.prepare_inputs(qd, kd, *zd, comba_d=comba_d, **P, **kw)
    torch.cuda.synchronize()
    qh, kh, al, be, mu, eta = [t.cpu().double().numpy() for t in out]
    rq, rk = G.prepare_qk(q.double().numpy(), k.double().numpy(), comba_d)
    ra, rb, rm, re = G.gates(*[t.double().numpy() for t in z], **P)
    tol_qk = 4e-3 if dtype == "bf16" else 1e-5
    errs = dict(q=_rel(qh, rq), k=_rel(kh, rk), alpha=_rel(al, ra), beta=_rel(be, rb),
                mu=_rel(mu, rm), eta=_rel(eta, re))
    assert errs["q"] <= tol_qk and errs["k"] <= tol_qk, errs
    for n in ("alpha", "beta", "mu", "eta"):
        assert errs[n] <= 1e-5, errs
    assert np.all(kh[1, 0] == 0)
    if comba_d == 0.5:
        assert np.all(qh[2, 0] == 0)
    assert np.all(al + be <= 1 + 1e-6)
    return errs


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_prepare_inputs_small(dtype, D):
    _check(37, 3, D, dtype, seed=1)


def test_prepare_inputs_in_place():
    _check(20, 2, 128, "bf16", seed=2, in_place=True)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_prepare_inputs_whole_tiles_and_tail(dtype, D):
    """Several whole 16 KiB tiles stream through shared memory; the rows after
    the last whole tile take the one-shot kernel."""
    _check(301, 3, D, dtype, seed=6)


def test_prepare_inputs_in_place_streaming():
    _check(500, 2, 128, "bf16", seed=7, in_place=True)


def test_prepare_inputs_no_correction():
    _check(20, 2, 128, "fp32", seed=3, comba_d=0.0)


def test_prepare_inputs_400m_shapes():
    """The prefill_400m token count and heads (8 x 2048 tokens, 8 heads)."""
    _check(16384, 8, 128, "bf16", seed=4)


def test_prepare_inputs_feed_the_forward():
    """The prepared inputs drive mdn_chunk_fwd as given (gates in range)."""
    import momentum_delta_rule_gb300 as mdn
    q, k, z = _inputs(2 * 130, 2, 128, "bf16", seed=5, zero_rows=False)
    qh, kh, al, be, mu, eta = mdn.prepare_inputs(q.cuda(), k.cuda(), *[t.cuda() for t in z], **P)
    v = torch.randn(2, 130, 2, 128).to(torch.bfloat16).cuda()
    shape4, shape3 = (2, 130, 2, 128), (2, 130, 2)
    o, S, M = mdn.chunk_fwd(qh.reshape(shape4), kh.reshape(shape4), v, al.reshape(shape3),
                            mu.reshape(shape3), eta.reshape(shape3), be.reshape(shape3))
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all() and torch.isfinite(M).all()
