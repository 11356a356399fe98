"""Pins of the gate parameterisation and query/key preparation oracle against
what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

from oracle import gates as G

P = dict(a=1.3, b=0.7, s=1.5, tau=2.0, log_mu_min=-2.0)


def _z(seed, n=4000, scale=4.0):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(n) * scale for _ in range(4)]


def test_alpha_plus_beta_at_most_one():
    """The frame's stated consequence of the coupled caps: alpha + beta <= 1."""
    al, be, mu, eta = G.gates(*_z(0), **P)
    assert np.all(al + be <= 1.0 + 1e-15)
    assert np.all(al > 0) and np.all(be >= 0)


def test_caps_closed_form():
    """cos^2(arctan x) = 1 / (1 + x^2): with z_alpha -> -inf (f -> 0) alpha
    reaches its cap 1 / (1 + s^2 eta^2), and beta's cap is the complement."""
    ze = np.linspace(-6, 6, 25)
    n = ze.size
    al, be, _, eta = G.gates(np.full(n, -60.0), np.full(n, 60.0), np.zeros(n), ze, **P)
    x2 = (P["s"] * eta) ** 2
    assert np.allclose(al, 1.0 / (1.0 + x2), rtol=1e-12, atol=0)
    assert np.allclose(be, x2 / (1.0 + x2), rtol=1e-12, atol=0)


def test_eta_range_and_centre():
    _, _, _, eta = G.gates(*_z(1), **P)
    assert np.all(eta > 0) and np.all(eta < 2)
    _, _, _, e0 = G.gates(np.zeros(1), np.zeros(1), np.zeros(1), np.zeros(1), **P)
    assert e0[0] == 1.0


def test_decay_function_values():
    """f(-b) = -a log 2; f -> -a (z + b) for large z; mu's floor applies."""
    n = 3
    z = np.array([-P["b"], 40.0 - P["b"], -80.0])
    al, _, mu, eta = G.gates(z, np.zeros(n), z, np.zeros(n), **P)
    cap = 1.0 / (1.0 + (P["s"] * eta) ** 2)
    assert np.isclose(np.log(al[0] / cap[0]), -P["a"] * np.log(2.0), rtol=1e-12)
    assert np.isclose(np.log(al[1] / cap[1]), -P["a"] * 40.0, rtol=1e-12)
    assert np.isclose(al[2], cap[2], rtol=1e-12)
    assert np.isclose(mu[0], np.exp(max(-P["a"] * np.log(2.0), P["log_mu_min"])), rtol=1e-12)
    assert np.isclose(mu[1], np.exp(P["log_mu_min"]), rtol=1e-12)     # floored
    assert np.isclose(mu[2], 1.0, rtol=1e-12)
    _, _, mu_all, _ = G.gates(*_z(2), **P)
    assert np.all(np.log(mu_all) >= P["log_mu_min"] - 1e-12)


def test_beta_is_sigmoid_of_projection_times_cap():
    n = 5
    zb = np.array([-3.0, -0.5, 0.0, 0.5, 3.0])
    _, be, _, eta = G.gates(np.zeros(n), zb, np.zeros(n), np.zeros(n), **P)
    cap = 1.0 - 1.0 / (1.0 + (P["s"] * eta) ** 2)
    assert np.allclose(be, cap / (1.0 + np.exp(-zb)), rtol=1e-12)


def test_qk_unit_norm_and_direction():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((50, 4, 16))
    k = rng.standard_normal((50, 4, 16))
    qh, kh = G.prepare_qk(q, k, 0.3)
    assert np.allclose(np.linalg.norm(qh, axis=-1), 1.0)
    assert np.allclose(np.linalg.norm(kh, axis=-1), 1.0)
    # q_hat is parallel to q - 0.3 k: their cross terms vanish
    w = q - 0.3 * k
    cos = np.sum(qh * w, -1) / np.linalg.norm(w, axis=-1)
    assert np.allclose(cos, 1.0)
    qh0, kh0 = G.prepare_qk(q, k, 0.0)
    assert np.allclose(qh0, q / np.linalg.norm(q, axis=-1, keepdims=True))
    assert np.allclose(kh0, kh)


def test_qk_zero_rows_stay_zero():
    q = np.zeros((2, 1, 8))
    k = np.zeros((2, 1, 8))
    k[1, 0, 3] = 2.0
    q[1, 0, 3] = 0.5                       # q - 0.25 k = 0
    qh, kh = G.prepare_qk(q, k, 0.25)
    assert np.all(qh == 0)
    assert np.all(kh[0] == 0) and kh[1, 0, 3] == 1.0


@pytest.mark.parametrize("mistake", ["sin_for_cos", "no_tau", "mu_no_floor", "beta_no_cap"])
def test_planted_mistakes_are_caught(mistake):
    """A copy of the gate formulas with one planted mistake fails a pin."""
    def bad(za, zb, zm, ze, a, b, s, tau, log_mu_min):
        eta = 1.0 + np.tanh(ze / (1.0 if mistake == "no_tau" else tau))
        th = np.arctan(s * eta)
        amax = (np.sin(th) if mistake == "sin_for_cos" else np.cos(th)) ** 2
        bmax = np.sin(th) ** 2
        f = lambda z: -a * G.softplus(z + b)
        al = np.exp(f(za)) * amax
        be = G.sigmoid(zb) * (1.0 if mistake == "beta_no_cap" else bmax)
        lm = f(zm) if mistake == "mu_no_floor" else np.maximum(f(zm), log_mu_min)
        return al, be, np.exp(lm), eta
    za, zb, zm, ze = _z(4)
    al, be, mu, eta = bad(za, zb, zm, ze, **P)
    ok = np.all(al + be <= 1 + 1e-15)
    x2 = (P["s"] * eta) ** 2
    a0, _, _, e0 = bad(np.full(3, -60.0), np.zeros(3), np.zeros(3), np.array([-1.0, 0.0, 1.0]), **P)
    ok &= np.allclose(a0, 1.0 / (1.0 + (P["s"] * e0) ** 2), rtol=1e-12)
    ok &= np.all(np.log(mu) >= P["log_mu_min"] - 1e-12)
    _, _, _, e1 = bad(np.zeros(1), np.zeros(1), np.zeros(1), np.array([2.0]), **P)
    ok &= np.isclose(e1[0], 1.0 + np.tanh(2.0 / P["tau"]))
    assert not ok, mistake
