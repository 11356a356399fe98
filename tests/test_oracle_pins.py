"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Each check is written as a function of a ``forward`` implementation so that it
can be run both against the oracle (must pass) and against copies of the
recurrence with a planted mistake (must fail): a dropped term, a wrong sign,
a wrong index, a transposed operand.  The planted copies live only in this
file and only on the CPU.
"""
import os

import numpy as np
import pytest

from oracle import chunkwise, coefficients as coef, recurrence

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers

def _rand_inputs(rng, T, H, dk, dv, mu_zero=False, alpha_one=False,
                 eta_one=False, beta_mode="rand", state=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    alpha = np.ones((T, H)) if alpha_one else np.exp(-rng.uniform(0, 0.3, (T, H)))
    mu = np.zeros((T, H)) if mu_zero else rng.uniform(0, 0.9, (T, H))
    eta = np.ones((T, H)) if eta_one else 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    if beta_mode == "rand":
        beta = rng.uniform(0.2, 1.0, (T, H))
    else:
        beta = None
    S0 = rng.standard_normal((1, H, dk, dv)) * 0.3 if state else None
    M0 = rng.standard_normal((1, H, dk, dv)) * 0.3 if state else None
    return dict(q=q, k=k, v=v, alpha=alpha, mu=mu, eta=eta, beta=beta,
                S0=S0, M0=M0)


def oracle_forward(x):
    return recurrence.forward(x["q"], x["k"], x["v"], x["alpha"], x["mu"],
                              x["eta"], x["beta"], x["S0"], x["M0"],
                              cu_seqlens=[0, x["q"].shape[0]])


def planted_forward(mistake):
    """A copy of the recurrence with one planted mistake (single sequence)."""
    def fwd(x):
        q, k, v = x["q"], x["k"], x["v"]
        T, H, dk = q.shape
        dv = v.shape[-1]
        beta = x["beta"] if x["beta"] is not None else np.ones((T, H))
        o = np.zeros((T, H, dv))
        S_T = np.zeros((1, H, dk, dv))
        M_T = np.zeros((1, H, dk, dv))
        for h in range(H):
            S = x["S0"][0, h].copy() if x["S0"] is not None else np.zeros((dk, dv))
            M = x["M0"][0, h].copy() if x["M0"] is not None else np.zeros((dk, dv))
            for t in range(T):
                a, m, e, b = x["alpha"][t, h], x["mu"][t, h], x["eta"][t, h], beta[t, h]
                kt, qt, vt = k[t, h], q[t, h], v[t, h]
                M_prev = M.copy()
                if mistake == "no_alpha_in_residual":
                    vr = vt - S.T @ kt
                else:
                    vr = vt - S.T @ (a * kt)
                if mistake == "momentum_sign":
                    M = m * M + e * np.outer(kt, vr)
                elif mistake == "no_eta":
                    M = m * M - np.outer(kt, vr)
                elif mistake == "mu_index":          # uses last step's mu
                    mp = x["mu"][t - 1, h] if t > 0 else m
                    M = mp * M - e * np.outer(kt, vr)
                else:
                    M = m * M - e * np.outer(kt, vr)
                if mistake == "old_momentum":        # S update with M_{t-1}
                    S = a * S - b * M_prev
                elif mistake == "no_beta":
                    S = a * S - M
                else:
                    S = a * S - b * M
                if mistake == "transposed_read" and dk == dv:
                    o[t, h] = S @ qt
                else:
                    o[t, h] = S.T @ qt
            S_T[0, h] = S
            M_T[0, h] = M
        return o, S_T, M_T
    return fwd


MISTAKES = ["no_alpha_in_residual", "momentum_sign", "no_eta", "mu_index",
            "old_momentum", "no_beta", "transposed_read"]


# --------------------------------------------------------------------------
# pin functions: return True when ``fwd`` satisfies the pinned property

def pin_gdn_reduction(fwd, seed=0):
    """mu = 0: the gated delta rule with write strength beta*eta.

    Reading notes section 1 (GDN equation) and section 2.2: setting mu = 0,
    eta = 1 recovers GDN; with general eta the write is scaled by beta*eta.
    Written here in its own textbook form, one state only.
    """
    rng = np.random.default_rng(seed)
    x = _rand_inputs(rng, 9, 2, 4, 4, mu_zero=True)
    o, S_T, _ = fwd(x)
    T, H, _ = x["q"].shape
    ok = True
    for h in range(H):
        S = x["S0"][0, h].copy()
        for t in range(T):
            a, e, b = x["alpha"][t, h], x["eta"][t, h], x["beta"][t, h]
            kt = x["k"][t, h]
            err = x["v"][t, h] - a * (S.T @ kt)
            S = a * S + b * e * np.outer(kt, err)
            ok &= np.allclose(o[t, h], S.T @ x["q"][t, h], atol=1e-12)
        ok &= np.allclose(S_T[0, h], S, atol=1e-12)
    return bool(ok)


def pin_deltanet_reduction(fwd, seed=1):
    """mu = 0, alpha = 1, eta = 1: DeltaNet, written in the other page's
    orientation (the state maps keys to values: S' = S^T in R^{dv x dk},
    S'_t = S'_{t-1} + beta (v - S'_{t-1} k) k^T, o = S' q)."""
    rng = np.random.default_rng(seed)
    x = _rand_inputs(rng, 8, 2, 3, 5, mu_zero=True, alpha_one=True, eta_one=True)
    o, S_T, _ = fwd(x)
    ok = True
    for h in range(2):
        Sp = x["S0"][0, h].T.copy()          # dv x dk
        for t in range(8):
            kt, b = x["k"][t, h], x["beta"][t, h]
            Sp = Sp + b * np.outer(x["v"][t, h] - Sp @ kt, kt)
            ok &= np.allclose(o[t, h], Sp @ x["q"][t, h], atol=1e-12)
        ok &= np.allclose(S_T[0, h], Sp.T, atol=1e-12)
    return bool(ok)


def pin_two_step(fwd, a2, b1, b2, m2, seed=2):
    """S_2 = (alpha_2 beta_1 + beta_2 mu_2) khat_1 vres_1^T + beta_2 khat_2 vres_2^T
    from S_0 = M_0 = 0 (slides "One error can affect several future writes")."""
    rng = np.random.default_rng(seed)
    dk, dv = 3, 4
    k = rng.standard_normal((2, 1, dk))
    v = rng.standard_normal((2, 1, dv))
    q = rng.standard_normal((2, 1, dk))
    eta = rng.uniform(0.3, 1.0, (2, 1))
    alpha = np.array([[rng.uniform(0.5, 1.0)], [a2]])
    mu = np.array([[rng.uniform(0.0, 1.0)], [m2]])
    beta = np.array([[b1], [b2]])
    x = dict(q=q, k=k, v=v, alpha=alpha, mu=mu, eta=eta, beta=beta,
             S0=None, M0=None)
    _, S_T, _ = fwd(x)
    kh1, kh2 = eta[0, 0] * k[0, 0], eta[1, 0] * k[1, 0]
    vres1 = v[0, 0]                                  # S_0 = 0
    S1 = b1 * np.outer(kh1, vres1)                   # one step from zero
    vres2 = v[1, 0] - a2 * (S1.T @ k[1, 0])
    w = a2 * b1 + b2 * m2
    S2 = w * np.outer(kh1, vres1) + b2 * np.outer(kh2, vres2)
    return bool(np.allclose(S_T[0, 0], S2, atol=1e-12))


def transition_matrix(a, m, b, e, k):
    """A_t of reading notes section 2.7 / slides backup "the full spectrum"."""
    dk = k.shape[0]
    I = np.eye(dk)
    kk = np.outer(k, k)
    return np.block([[a * I - a * b * e * kk, -b * m * I],
                     [a * e * kk, m * I]])


def pin_transition(fwd, seed=3):
    """One step equals A_t [S; M] + [beta eta k v^T; -eta k v^T]."""
    rng = np.random.default_rng(seed)
    ok = True
    for _ in range(4):
        x = _rand_inputs(rng, 1, 1, 5, 3)
        _, S1, M1 = fwd(x)
        a, m, e, b = (x["alpha"][0, 0], x["mu"][0, 0], x["eta"][0, 0],
                      x["beta"][0, 0])
        kt, vt = x["k"][0, 0], x["v"][0, 0]
        A = transition_matrix(a, m, b, e, kt)
        drive = np.vstack([b * e * np.outer(kt, vt), -e * np.outer(kt, vt)])
        SM = A @ np.vstack([x["S0"][0, 0], x["M0"][0, 0]]) + drive
        ok &= np.allclose(S1[0, 0], SM[:5], atol=1e-12)
        ok &= np.allclose(M1[0, 0], SM[5:], atol=1e-12)
    return bool(ok)


def pin_second_order(fwd, seed=4):
    """Eliminating M (beta_{t-1} != 0):
    S_t = [(alpha_t + beta_t mu_t / beta_{t-1}) I - alpha_t beta_t eta_t k k^T] S_{t-1}
          - (beta_t mu_t alpha_{t-1} / beta_{t-1}) S_{t-2} + beta_t eta_t k v_t^T
    (slides backup "eliminating momentum reveals the second-order rule")."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 7, 4, 3
    x = _rand_inputs(rng, T, 1, dk, dv)
    states = [x["S0"][0, 0]]
    for t in range(1, T + 1):
        sub = {kk: (vv[:t] if kk not in ("S0", "M0") and vv is not None else vv)
               for kk, vv in x.items()}
        _, S_t, _ = fwd(sub)
        states.append(S_t[0, 0])
    ok = True
    I = np.eye(dk)
    for t in range(2, T + 1):          # 1-based token index t
        i, ip = t - 1, t - 2           # 0-based rows of token t and t-1
        a, m, e, b = x["alpha"][i, 0], x["mu"][i, 0], x["eta"][i, 0], x["beta"][i, 0]
        ap, bp = x["alpha"][ip, 0], x["beta"][ip, 0]
        kt, vt = x["k"][i, 0], x["v"][i, 0]
        lhs = states[t]
        rhs = (((a + b * m / bp) * I - a * b * e * np.outer(kt, kt)) @ states[t - 1]
               - (b * m * ap / bp) * states[t - 2] + b * e * np.outer(kt, vt))
        ok &= np.allclose(lhs, rhs, atol=1e-10)
    return bool(ok)


# --------------------------------------------------------------------------
# the oracle satisfies every pin

def test_gdn_reduction():
    assert pin_gdn_reduction(oracle_forward)


def test_deltanet_reduction():
    assert pin_deltanet_reduction(oracle_forward)


def pin_deltanet_residual(seed=5):
    """The per-token residual the forward can save ("Backward computation"
    frame: save the corrected values) reduces, for mu = 0, alpha = 1,
    eta = 1, to DeltaNet's prediction error v_t - S'_{t-1} k_t in the other
    page's key-to-value orientation; checked against that form written out,
    with a nonzero initial state and a state carried over a sequence split."""
    rng = np.random.default_rng(seed)
    x = _rand_inputs(rng, 9, 2, 3, 5, mu_zero=True, alpha_one=True, eta_one=True)
    _, _, _, vres = recurrence.forward(x["q"], x["k"], x["v"], x["alpha"], x["mu"],
                                       x["eta"], x["beta"], x["S0"], x["M0"],
                                       cu_seqlens=[0, 9], return_vres=True)
    ok = True
    for h in range(2):
        Sp = x["S0"][0, h].T.copy()
        for t in range(9):
            kt, b = x["k"][t, h], x["beta"][t, h]
            err = x["v"][t, h] - Sp @ kt
            ok &= np.allclose(vres[t, h], err, atol=1e-12)
            Sp = Sp + b * np.outer(err, kt)
    return bool(ok)


def test_deltanet_residual():
    assert pin_deltanet_residual()


def test_residual_output_does_not_change_the_forward():
    rng = np.random.default_rng(6)
    x = _rand_inputs(rng, 11, 2, 4, 3)
    a = oracle_forward(x)
    b = recurrence.forward(x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"],
                           x["beta"], x["S0"], x["M0"], cu_seqlens=[0, 11],
                           return_vres=True)
    for u, w in zip(a, b[:3]):
        assert np.array_equal(u, w)
    assert b[3].shape == x["v"].shape


def test_two_step_worked_example_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "two_step_weight.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) >= 4
    for a2, b1, b2, m2, w in rows:
        a2, b1, b2, m2, w = map(float, (a2, b1, b2, m2, w))
        assert a2 * b1 + b2 * m2 == w          # the fixture is the printed form
        assert pin_two_step(oracle_forward, a2, b1, b2, m2)


def test_transition_matrix_form():
    assert pin_transition(oracle_forward)


def test_transition_spectrum():
    """Spec(A_t) = {alpha (dk-1 times), mu (dk-1 times), lambda_+-}, with
    r = alpha + mu - alpha beta eta and lambda = (r +- sqrt(r^2 - 4 alpha mu))/2
    for a unit key (slides "Momentum permits damped oscillatory modes",
    Appendix F Eq. (60))."""
    rng = np.random.default_rng(5)
    for dk in (2, 3, 5):
        for _ in range(5):
            a, m = rng.uniform(0.1, 1.0), rng.uniform(0.0, 1.0)
            b, e = rng.uniform(0.0, 1.0), rng.uniform(0.0, 2.0)
            k = rng.standard_normal(dk)
            k /= np.linalg.norm(k)
            ev = np.linalg.eigvals(transition_matrix(a, m, b, e, k))
            r = a + m - a * b * e
            disc = np.sqrt(complex(r * r - 4 * a * m))
            expect = np.array([a] * (dk - 1) + [m] * (dk - 1)
                              + [(r + disc) / 2, (r - disc) / 2], dtype=complex)
            got = np.sort_complex(np.round(ev, 9))
            exp = np.sort_complex(np.round(expect, 9))
            np.testing.assert_allclose(got, exp, atol=1e-7)


def test_second_order_identity():
    assert pin_second_order(oracle_forward)


@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistake_is_caught(mistake):
    """Every planted mistake in a copy of the recurrence fails some pin."""
    fwd = planted_forward(mistake)
    results = [pin_gdn_reduction(fwd), pin_deltanet_reduction(fwd),
               pin_transition(fwd), pin_second_order(fwd),
               all(pin_two_step(fwd, *c) for c in
                   [(0.5, 0.25, 1.0, 0.75), (0.75, 0.5, 0.5, 0.5)])]
    assert not all(results), mistake


def test_planted_copy_without_mistake_passes():
    """The pins are not trivially failing: the unplanted copy passes them."""
    fwd = planted_forward("none")
    assert pin_gdn_reduction(fwd) and pin_deltanet_reduction(fwd)
    assert pin_transition(fwd) and pin_second_order(fwd)


# --------------------------------------------------------------------------
# chunkwise algebra: exact reformulation of the recurrence

@pytest.mark.parametrize("C", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chunkwise_equals_recurrence_bruteforce(C, seed):
    """'Chunking is an exact algebraic reformulation' (slides, chunk-output
    frame; reading notes 2.5): equal to ~1e-12 on tiny inputs."""
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 13))
    dk, dv = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    x = _rand_inputs(rng, T, 2, dk, dv)
    o, S, M = oracle_forward(x)
    o2, S2, M2 = chunkwise.chunk_forward_packed(
        x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
        x["S0"], x["M0"], [0, T], C=C)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(S2, S, atol=1e-12)
    np.testing.assert_allclose(M2, M, atol=1e-12)


@pytest.mark.parametrize("gamma_fn", [coef.gamma_column_recurrence,
                                      coef.gamma_triple_sum])
def test_chunkwise_mu_zero_and_beta_zero(gamma_fn):
    """mu = 0 and beta = 0 entries must not produce NaN (the recurrence
    permits mu = 0; slides' ablation frame notes the paper's kernel did not)."""
    rng = np.random.default_rng(7)
    T = 12
    x = _rand_inputs(rng, T, 1, 3, 3)
    x["mu"][::3] = 0.0
    x["beta"][1::4] = 0.0
    o, S, M = oracle_forward(x)
    o2, S2, M2 = chunkwise.chunk_forward_packed(
        x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
        x["S0"], x["M0"], [0, T], C=8, gamma_fn=gamma_fn)
    assert np.isfinite(o2).all()
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(S2, S, atol=1e-12)
    np.testing.assert_allclose(M2, M, atol=1e-12)


def test_row_shift_is_required():
    """Deleting Gamma's diagonal instead of shifting it down one row gives the
    wrong residual coefficients (slides backup frame; golden 3x3 pattern)."""
    rng = np.random.default_rng(8)
    x = _rand_inputs(rng, 8, 1, 3, 3)
    o, _, _ = oracle_forward(x)
    o_bad, _, _ = chunkwise.chunk_forward_packed(
        x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
        x["S0"], x["M0"], [0, 8], C=4, shift="strict")
    assert np.abs(o_bad - o).max() > 1e-3


def test_gamma_shift_golden_pattern():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "gamma_row_shift_3x3.txt"))
             if l.strip() and not l.startswith("#")]
    gi = lines.index(["Gamma"])
    si = lines.index(["Gamma_shifted"])
    pat_G = lines[gi + 1:gi + 4]
    pat_S = lines[si + 1:si + 4]
    rng = np.random.default_rng(9)
    a, m, b = rng.uniform(0.5, 1, 3), rng.uniform(0, 1, 3), rng.uniform(0.2, 1, 3)
    cv = coef.chunk_vectors(a, m, b)
    G, Gm = cv["Gamma"], cv["Gamma_m"]

    def val(tok):
        if tok == "0":
            return 0.0
        return G[int(tok[1]) - 1, int(tok[2]) - 1]
    for i in range(3):
        for j in range(3):
            assert G[i, j] == val(pat_G[i][j])
            assert Gm[i, j] == val(pat_S[i][j])


def test_state_passing_split_invariance():
    """fwd(x[0:T]) equals fwd(x[T1:T]) started from fwd(x[0:T1])'s states
    (chunk carry, slides Appendix C Eqs. (40)-(42))."""
    rng = np.random.default_rng(10)
    T, T1 = 11, 4
    x = _rand_inputs(rng, T, 2, 3, 4)
    o, S, M = oracle_forward(x)
    first = {kk: (vv[:T1] if kk not in ("S0", "M0") else vv) for kk, vv in x.items()}
    o1, S1, M1 = oracle_forward(first)
    second = {kk: (vv[T1:] if kk not in ("S0", "M0") else vv) for kk, vv in x.items()}
    second["S0"], second["M0"] = S1, M1
    o2, S2, M2 = oracle_forward(second)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, atol=1e-13)
    np.testing.assert_allclose(S2, S, atol=1e-13)
    np.testing.assert_allclose(M2, M, atol=1e-13)


def test_varlen_packing_resets_state():
    rng = np.random.default_rng(11)
    lens = [3, 0, 5, 1]
    T = sum(lens)
    x = _rand_inputs(rng, T, 2, 3, 3, state=False)
    cu = np.cumsum([0] + lens)
    o, S, M = recurrence.forward(x["q"], x["k"], x["v"], x["alpha"], x["mu"],
                                 x["eta"], x["beta"], cu_seqlens=cu)
    for s, L in enumerate(lens):
        sl = slice(cu[s], cu[s + 1])
        sub = {kk: (vv[sl] if vv is not None else None) for kk, vv in x.items()}
        o1, S1, M1 = recurrence.forward(sub["q"], sub["k"], sub["v"],
                                        sub["alpha"], sub["mu"], sub["eta"],
                                        sub["beta"], cu_seqlens=[0, L])
        np.testing.assert_allclose(o[sl], o1, atol=1e-14)
        np.testing.assert_allclose(S[s], S1[0], atol=1e-14)
        np.testing.assert_allclose(M[s], M1[0], atol=1e-14)
    assert np.all(S[1] == 0) and np.all(M[1] == 0)       # empty sequence


def test_decode_steps_equal_forward():
    """Decoding uses the same token recurrence (slides chunk-output frame)."""
    rng = np.random.default_rng(12)
    T, N, H, d = 5, 3, 2, 4
    xs = [_rand_inputs(rng, T, H, d, d) for _ in range(N)]
    S = np.stack([x["S0"][0] for x in xs])
    M = np.stack([x["M0"][0] for x in xs])
    S_ref, M_ref = S.copy(), M.copy()
    for t in range(T):
        q = np.stack([x["q"][t] for x in xs])
        k = np.stack([x["k"][t] for x in xs])
        v = np.stack([x["v"][t] for x in xs])
        g = {n: np.stack([x[n][t] for x in xs]) for n in ("alpha", "mu", "eta", "beta")}
        o, S, M = recurrence.decode_step(q, k, v, g["alpha"], g["mu"], g["eta"],
                                         S, M, beta=g["beta"])
    for n, x in enumerate(xs):
        o_f, S_f, M_f = oracle_forward(x)
        np.testing.assert_allclose(o[n], o_f[-1], atol=1e-13)
        np.testing.assert_allclose(S[n], S_f[0], atol=1e-13)
        np.testing.assert_allclose(M[n], M_f[0], atol=1e-13)


@pytest.mark.parametrize("C", [16, 32, 64])
def test_chunkwise_at_kernel_chunk_sizes_packed(C):
    """The chunkwise form at the kernel's chunk size (64) and below, over packed
    sequences with full chunks, ragged tails, an empty sequence, per-sequence
    initial states and zero momentum gates, equals the token recurrence to
    rounding (slides Appendix C, chunk carry Eqs. (40)-(42); partial last
    chunk per the reading that each sequence is chunked from its own start)."""
    rng = np.random.default_rng(13)
    lens = [70, 0, 64, 17, 150]
    T = sum(lens)
    x = _rand_inputs(rng, T, 2, 8, 6)
    x["mu"][::7] = 0.0
    cu = np.cumsum([0] + lens)
    S0 = rng.standard_normal((len(lens), 2, 8, 6)) * 0.3
    M0 = rng.standard_normal((len(lens), 2, 8, 6)) * 0.3
    o, S, M = recurrence.forward(x["q"], x["k"], x["v"], x["alpha"], x["mu"],
                                 x["eta"], x["beta"], S0, M0, cu_seqlens=cu)
    o2, S2, M2 = chunkwise.chunk_forward_packed(
        x["q"], x["k"], x["v"], x["alpha"], x["mu"], x["eta"], x["beta"],
        S0, M0, cu, C=C)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(S2, S, atol=1e-12)
    np.testing.assert_allclose(M2, M, atol=1e-12)
    np.testing.assert_array_equal(S2[1], S0[1])            # empty sequence
    np.testing.assert_array_equal(M2[1], M0[1])
