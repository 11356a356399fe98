"""Pins of the fp64 backward oracle (``oracle/backward.py``).

The pages give no gradient formulas, only the storage policy for training
(slides, "Backward computation" block: save the residuals, rebuild the
states, do not keep every state pair).  The gradient is therefore pinned to
the mathematics that defines it: central finite differences of the forward
oracle (the C token recurrence, written independently), entry by entry on a
tiny case and along random directions on packed sequences; and the rebuilt
states to the forward's own states.  Planted mistakes show that the
difference check fails when a term is wrong.  The chunkwise gradient
(``oracle/chunkwise_backward.py``) is pinned to the token-level sweep.
"""
import numpy as np
import pytest

from oracle import backward as bwd, chunkwise_backward as cbwd, recurrence

NAMES = ("q", "k", "v", "alpha", "mu", "eta", "beta", "S0", "M0")


def _inputs(rng, lens, H, dk, dv, mu_zero_every=0):
    T = sum(lens)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    x = dict(q=q, k=k, v=rng.standard_normal((T, H, dv)),
             alpha=np.exp(-rng.uniform(0, 0.3, (T, H))),
             mu=rng.uniform(0, 0.9, (T, H)),
             eta=1 / (1 + np.exp(-rng.standard_normal((T, H)))),
             beta=rng.uniform(0.2, 1.0, (T, H)),
             S0=rng.standard_normal((len(lens), H, dk, dv)) * 0.3,
             M0=rng.standard_normal((len(lens), H, dk, dv)) * 0.3)
    if mu_zero_every:
        x["mu"][::mu_zero_every] = 0.0
    return x, np.cumsum([0] + list(lens))


def _weights(rng, x, n_seq):
    T, H, dv = x["v"].shape
    dk = x["q"].shape[2]
    return (rng.standard_normal((T, H, dv)),
            rng.standard_normal((n_seq, H, dk, dv)),
            rng.standard_normal((n_seq, H, dk, dv)))


def _loss(x, cu, W):
    o, S, M = recurrence.forward(x["q"], x["k"], x["v"], x["alpha"], x["mu"],
                                 x["eta"], x["beta"], x["S0"], x["M0"],
                                 cu_seqlens=cu)
    return float((o * W[0]).sum() + (S * W[1]).sum() + (M * W[2]).sum())


def _directional_errors(grad_fn, x, cu, W, rng, h=1e-6):
    g = grad_fn(x, cu, W)
    errs = {}
    for name in NAMES:
        E = rng.standard_normal(x[name].shape)
        xp, xm = dict(x), dict(x)
        xp[name] = x[name] + h * E
        xm[name] = x[name] - h * E
        fd = (_loss(xp, cu, W) - _loss(xm, cu, W)) / (2 * h)
        an = float((g["d" + name] * E).sum())
        errs[name] = abs(fd - an) / max(1.0, abs(fd))
    return errs


def _oracle_grad(x, cu, W):
    return bwd.backward(**x, do=W[0], dS_T=W[1], dM_T=W[2], cu_seqlens=cu)


@pytest.mark.parametrize("seed,lens,mu0", [(0, [7], 0), (1, [5, 0, 9, 1], 3),
                                           (2, [12, 4], 2)])
def test_gradients_match_central_differences(seed, lens, mu0):
    """Every input's gradient along a random direction equals the central
    difference of the forward oracle (packed sequences, an empty one, zero
    momentum gates)."""
    rng = np.random.default_rng(200 + seed)
    x, cu = _inputs(rng, lens, 2, 3, 4, mu_zero_every=mu0)
    W = _weights(rng, x, len(lens))
    errs = _directional_errors(_oracle_grad, x, cu, W, rng)
    assert max(errs.values()) < 1e-7, errs


def test_every_gradient_entry_on_a_tiny_case():
    """Entry-by-entry central differences, T = 3, one head, dk = dv = 2."""
    rng = np.random.default_rng(210)
    x, cu = _inputs(rng, [3], 1, 2, 2)
    W = _weights(rng, x, 1)
    g = _oracle_grad(x, cu, W)
    h = 1e-6
    for name in NAMES:
        flat = x[name].reshape(-1)
        for e in range(flat.size):
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[name].reshape(-1)[e] += h
            xm[name].reshape(-1)[e] -= h
            fd = (_loss(xp, cu, W) - _loss(xm, cu, W)) / (2 * h)
            an = g["d" + name].reshape(-1)[e]
            assert abs(fd - an) < 1e-7 * max(1.0, abs(fd)), (name, e, fd, an)


def test_beta_absent_means_one():
    """beta = None is beta = 1: same gradients, and dbeta is the gradient at 1."""
    rng = np.random.default_rng(220)
    x, cu = _inputs(rng, [6], 2, 3, 3)
    W = _weights(rng, x, 1)
    x1 = dict(x, beta=np.ones_like(x["beta"]))
    g1 = _oracle_grad(x1, cu, W)
    gn = _oracle_grad(dict(x, beta=None), cu, W)
    for kk in g1:
        np.testing.assert_array_equal(gn[kk], g1[kk])


def test_packed_gradients_are_per_sequence():
    """Packing restarts the state: each sequence's gradients are those of the
    sequence run alone."""
    rng = np.random.default_rng(230)
    lens = [4, 0, 6]
    x, cu = _inputs(rng, lens, 2, 3, 2)
    W = _weights(rng, x, len(lens))
    g = _oracle_grad(x, cu, W)
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        xs = {kk: (vv[sl] if kk not in ("S0", "M0") else vv[s:s + 1]) for kk, vv in x.items()}
        Ws = (W[0][sl], W[1][s:s + 1], W[2][s:s + 1])
        gs = bwd.backward(**xs, do=Ws[0], dS_T=Ws[1], dM_T=Ws[2], cu_seqlens=[0, lens[s]])
        for kk in ("dq", "dk", "dv", "dalpha", "dmu", "deta", "dbeta"):
            np.testing.assert_allclose(g[kk][sl], gs[kk], atol=1e-14)
        np.testing.assert_allclose(g["dS0"][s], gs["dS0"][0], atol=1e-14)
        np.testing.assert_allclose(g["dM0"][s], gs["dM0"][0], atol=1e-14)
    # an empty sequence passes the state adjoints straight through
    np.testing.assert_array_equal(g["dS0"][1], W[1][1])
    np.testing.assert_array_equal(g["dM0"][1], W[2][1])


def test_rebuilt_states_equal_the_forward():
    """The storage policy of the slides' backward block: from the saved
    residuals and a segment's entry states, M' = mu M - eta k vres^T and
    S' = alpha S - beta M' give back the forward's states, here the final
    states of the C oracle, also when the entry states come from splitting
    the sequence."""
    rng = np.random.default_rng(240)
    x, cu = _inputs(rng, [11], 2, 4, 3)
    o, S_T, M_T, vres = recurrence.forward(
        x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
        x["S0"], x["M0"], cu_seqlens=cu, return_vres=True)
    S_all, M_all = bwd.rebuild_states(x["k"], x["alpha"], x["mu"], x["eta"],
                                      x["beta"], vres, x["S0"][0], x["M0"][0])
    np.testing.assert_allclose(S_all[-1], S_T[0], atol=1e-13)
    np.testing.assert_allclose(M_all[-1], M_T[0], atol=1e-13)
    # outputs from the rebuilt states: o_t = S_t^T q_t
    np.testing.assert_allclose(np.einsum("thij,thi->thj", S_all[1:], x["q"]), o, atol=1e-13)
    # second half rebuilt from the state at the split point
    t1 = 5
    S2, M2 = bwd.rebuild_states(x["k"][t1:], x["alpha"][t1:], x["mu"][t1:],
                                x["eta"][t1:], x["beta"][t1:], vres[t1:],
                                S_all[t1], M_all[t1])
    np.testing.assert_allclose(S2[-1], S_T[0], atol=1e-13)
    np.testing.assert_allclose(M2[-1], M_T[0], atol=1e-13)


# --------------------------------------------------------------------------
# planted mistakes: the difference check must fail on each

def _planted(mistake):
    def grad(x, cu, W):
        if mistake == "dropped_state_adjoint":
            return bwd.backward(**x, do=W[0], dS_T=None, dM_T=W[2], cu_seqlens=cu)
        if mistake == "swapped_gates":
            return bwd.backward(**dict(x, alpha=x["mu"], mu=x["alpha"]), do=W[0],
                                dS_T=W[1], dM_T=W[2], cu_seqlens=cu)
        if mistake == "transposed_output_adjoint":
            xt = dict(x)
            return bwd.backward(**xt, do=W[0][:, ::-1].copy(), dS_T=W[1], dM_T=W[2],
                                cu_seqlens=cu)
        if mistake == "residual_sign":
            real = bwd._residuals
            try:
                bwd._residuals = lambda k, v, a, S: 2 * v - real(k, v, a, S)
                return bwd.backward(**x, do=W[0], dS_T=W[1], dM_T=W[2], cu_seqlens=cu)
            finally:
                bwd._residuals = real
        return _oracle_grad(x, cu, W)
    return grad


@pytest.mark.parametrize("mistake", ["dropped_state_adjoint", "swapped_gates",
                                     "transposed_output_adjoint", "residual_sign"])
def test_planted_mistake_fails_the_difference_check(mistake):
    rng = np.random.default_rng(250)
    x, cu = _inputs(rng, [6, 3], 2, 3, 3)
    W = _weights(rng, x, 2)
    errs = _directional_errors(_planted(mistake), x, cu, W, rng)
    assert max(errs.values()) > 1e-4, (mistake, errs)


def test_unplanted_copy_passes():
    rng = np.random.default_rng(250)
    x, cu = _inputs(rng, [6, 3], 2, 3, 3)
    W = _weights(rng, x, 2)
    errs = _directional_errors(_planted("none"), x, cu, W, rng)
    assert max(errs.values()) < 1e-7, errs


# --------------------------------------------------------------------------
# the chunkwise gradient (the algebra a chunked gradient pass follows)


@pytest.mark.parametrize("C,T", [(1, 5), (2, 7), (3, 12), (4, 9), (8, 20), (16, 37)])
@pytest.mark.parametrize("with_beta", [True, False])
def test_chunkwise_gradient_equals_token_sweep(C, T, with_beta):
    """Chunk by chunk (dense products per chunk, state adjoints carried
    backwards across chunks, gate partials through the chunk coefficients)
    equals the token-level reverse sweep to rounding, with zero momentum
    gates and a ragged last chunk."""
    rng = np.random.default_rng(300 + 7 * C + T)
    x, cu = _inputs(rng, [T], 1, 3, 4, mu_zero_every=3)
    if not with_beta:
        x["beta"] = None
    W = _weights(rng, x, 1)
    g = bwd.backward(**x, do=W[0], dS_T=W[1], dM_T=W[2], cu_seqlens=cu)
    gc = cbwd.chain_backward(
        x["q"][:, 0], x["k"][:, 0], x["v"][:, 0], x["alpha"][:, 0], x["mu"][:, 0],
        x["eta"][:, 0], None if x["beta"] is None else x["beta"][:, 0],
        x["S0"][0, 0], x["M0"][0, 0], W[0][:, 0], W[1][0, 0], W[2][0, 0], C=C)
    for name in ("dq", "dk", "dv", "dalpha", "dmu", "deta", "dbeta"):
        np.testing.assert_allclose(gc[name], g[name][:, 0], atol=1e-12, err_msg=name)
    np.testing.assert_allclose(gc["dS0"], g["dS0"][0, 0], atol=1e-12)
    np.testing.assert_allclose(gc["dM0"], g["dM0"][0, 0], atol=1e-12)


def test_chunkwise_gradient_with_strict_lower_gamma_fails(monkeypatch):
    """Deleting Gamma's diagonal instead of shifting its rows (the mistake the
    slides' backup frame warns about) breaks the chunkwise gradient too."""
    rng = np.random.default_rng(320)
    x, cu = _inputs(rng, [10], 1, 3, 3)
    W = _weights(rng, x, 1)
    g = bwd.backward(**x, do=W[0], dS_T=W[1], dM_T=W[2], cu_seqlens=cu)
    real = cbwd._coeffs

    def strict(a, m, b):
        c = real(a, m, b)
        c["Gm"] = np.tril(c["G"], -1)
        return c
    monkeypatch.setattr(cbwd, "_coeffs", strict)
    gc = cbwd.chain_backward(
        x["q"][:, 0], x["k"][:, 0], x["v"][:, 0], x["alpha"][:, 0], x["mu"][:, 0],
        x["eta"][:, 0], x["beta"][:, 0], x["S0"][0, 0], x["M0"][0, 0],
        W[0][:, 0], W[1][0, 0], W[2][0, 0], C=4)
    assert np.abs(gc["dk"] - g["dk"][:, 0]).max() > 1e-3


@pytest.mark.parametrize("n,seed", [(1, 0), (2, 1), (5, 2), (9, 3), (16, 4)])
def test_closed_form_gate_partials_equal_evaluation(n, seed):
    """The gate gradients as sums over Gamma's index triangle equal the exact
    gate-by-gate partials, for arbitrary coefficient adjoints, with zero and
    unit gates among them."""
    rng = np.random.default_rng(400 + seed)
    a = np.exp(-rng.uniform(0, 0.5, n))
    m = rng.uniform(0, 1, n)
    if n > 2:
        m[::2] = 0.0
    bt = rng.uniform(0, 1, n)
    a[-1] = 1.0
    c = cbwd._coeffs(a, m, bt)
    dc = {kk: rng.standard_normal(np.shape(vv)) for kk, vv in c.items()}
    dc = {kk: (float(vv) if np.ndim(vv) == 0 else vv) for kk, vv in dc.items()}
    ref = cbwd.gate_partials_by_evaluation(a, m, bt, dc)
    got = cbwd.gate_partials_closed_form(a, m, bt, dc)
    for r, g_ in zip(ref, got):
        np.testing.assert_allclose(g_, r, atol=1e-12)


@pytest.mark.parametrize("C,T", [(4, 13), (16, 37), (64, 150)])
def test_chunkwise_gradient_closed_form_equals_token_sweep(C, T):
    """At the kernel's chunk size too (two full chunks and a ragged one)."""
    rng = np.random.default_rng(500 + C)
    x, cu = _inputs(rng, [T], 1, 3, 4, mu_zero_every=4)
    W = _weights(rng, x, 1)
    g = bwd.backward(**x, do=W[0], dS_T=W[1], dM_T=W[2], cu_seqlens=cu)
    gc = cbwd.chain_backward(
        x["q"][:, 0], x["k"][:, 0], x["v"][:, 0], x["alpha"][:, 0], x["mu"][:, 0],
        x["eta"][:, 0], x["beta"][:, 0], x["S0"][0, 0], x["M0"][0, 0],
        W[0][:, 0], W[1][0, 0], W[2][0, 0], C=C,
        gate_partials=cbwd.gate_partials_closed_form)
    for name in ("dq", "dk", "dv", "dalpha", "dmu", "deta", "dbeta"):
        np.testing.assert_allclose(gc[name], g[name][:, 0], atol=1e-12, err_msg=name)


def test_chunkwise_gradient_packed_heads():
    """The packed, multi-head form (an empty sequence, ragged chunks) equals
    the token sweep over the same layout."""
    rng = np.random.default_rng(600)
    lens = [70, 0, 9, 33]
    x, cu = _inputs(rng, lens, 2, 3, 4, mu_zero_every=5)
    W = _weights(rng, x, len(lens))
    g = bwd.backward(**x, do=W[0], dS_T=W[1], dM_T=W[2], cu_seqlens=cu)
    gc = cbwd.chunk_backward_packed(**x, do=W[0], dS_T=W[1], dM_T=W[2],
                                    cu_seqlens=cu, C=16)
    for name in g:
        np.testing.assert_allclose(gc[name], g[name], atol=1e-12, err_msg=name)


@pytest.mark.parametrize("C", [3, 16, 64])
def test_chunkwise_gradient_forward_equals_recurrence(C):
    """The forward the chunkwise gradient differentiates (chunk by chunk,
    with its own saved quantities) is the recurrence itself."""
    rng = np.random.default_rng(700 + C)
    x, cu = _inputs(rng, [100], 1, 4, 3, mu_zero_every=6)
    o_ref, S_ref, M_ref = recurrence.forward(
        x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
        x["S0"], x["M0"], cu_seqlens=cu)
    S, M = x["S0"][0, 0], x["M0"][0, 0]
    o = []
    for s0 in range(0, 100, C):
        sl = slice(s0, min(s0 + C, 100))
        O, S, M, _ = cbwd._chunk_forward(
            x["q"][sl, 0], x["k"][sl, 0], x["v"][sl, 0], x["alpha"][sl, 0],
            x["mu"][sl, 0], x["eta"][sl, 0], x["beta"][sl, 0], S, M)
        o.append(O)
    np.testing.assert_allclose(np.concatenate(o), o_ref[:, 0], atol=1e-12)
    np.testing.assert_allclose(S, S_ref[0, 0], atol=1e-12)
    np.testing.assert_allclose(M, M_ref[0, 0], atol=1e-12)
