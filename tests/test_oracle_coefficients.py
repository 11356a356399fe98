"""Pins of the oracle's chunk coefficients (four independent evaluations)."""
import numpy as np
import pytest

from oracle import coefficients as coef


def _gates(rng, C, mu_lo=0.0, mu_hi=0.9):
    alpha = np.exp(-rng.uniform(0, 0.1, C))
    mu = rng.uniform(mu_lo, mu_hi, C)
    beta = rng.uniform(0.1, 1.0, C)
    return alpha, mu, beta


@pytest.mark.parametrize("C", [1, 2, 5, 8])
def test_forms_agree_on_small_chunks(C):
    rng = np.random.default_rng(C)
    a, m, b = _gates(rng, C, 0.3, 0.9)
    G0, b0 = coef.gamma_triple_sum(a, m, b)
    for fn in (coef.gamma_column_recurrence, coef.gamma_cumulative,
               coef.gamma_printed_log):
        G, bb = fn(a, m, b)
        np.testing.assert_allclose(G, G0, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(bb, b0, rtol=1e-9, atol=1e-12)


def test_column_recurrence_equals_definition_full_chunk():
    rng = np.random.default_rng(1)
    a, m, b = _gates(rng, 64)
    m[[5, 17, 40]] = 0.0
    G0, b0 = coef.gamma_triple_sum(a, m, b)
    G, bb = coef.gamma_column_recurrence(a, m, b)
    np.testing.assert_allclose(G, G0, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(bb, b0, rtol=1e-12, atol=1e-300)


def test_printed_form_on_well_conditioned_gates():
    """mu in [0.6, 1]: the printed log-domain form is accurate."""
    rng = np.random.default_rng(2)
    a, m, b = _gates(rng, 64, 0.6, 1.0)
    G0, b0 = coef.gamma_triple_sum(a, m, b)
    G, bb = coef.gamma_printed_log(a, m, b)
    np.testing.assert_allclose(G, G0, rtol=1e-7, atol=1e-12)
    np.testing.assert_allclose(bb, b0, rtol=1e-10)


def test_printed_form_cancels_for_small_mu():
    """mu ~ U(0, 0.9), beta = 1: the factor [1 - exp(l_{j-1} - l_i)] rounds
    away once the prefix log-sum-exp stops changing, so the printed form loses
    gamma_{j,j} = beta_j late in a 64-token chunk even in fp64.  This is why
    the stable evaluation (column recurrence / segment sums) is used."""
    rng = np.random.default_rng(3)
    a = np.exp(-rng.uniform(0, 0.1, 64))
    m = rng.uniform(0, 0.9, 64)
    b = np.ones(64)
    G, _ = coef.gamma_printed_log(a, m, b)
    diag_err = np.abs(np.diag(G) - 1.0)
    assert diag_err[:8].max() < 1e-9
    assert diag_err[-16:].max() > 1e-3


def test_diagonal_is_beta():
    """gamma_{i,i} = beta_i (reading notes 2.3, one-step relation)."""
    rng = np.random.default_rng(4)
    a, m, b = _gates(rng, 16)
    for fn in (coef.gamma_triple_sum, coef.gamma_column_recurrence):
        G, _ = fn(a, m, b)
        np.testing.assert_allclose(np.diag(G), b, rtol=1e-14)
        assert np.all(np.triu(G, 1) == 0)


def test_b_is_gamma_of_an_origin_before_the_chunk():
    """b_i = abar_i c_i is gamma_{i,0} with mubar_0 = 1: prepend a token with
    beta_0 = 0 and any alpha_0; column 0 of the extended Gamma is then b
    shifted by one (reading notes 2.3, abar_0 = mubar_0 = 1, c_0 = b_0 = 0)."""
    rng = np.random.default_rng(5)
    a, m, b = _gates(rng, 10)
    _, b_ref = coef.gamma_triple_sum(a, m, b)
    a_ext = np.concatenate([[0.77], a])
    m_ext = np.concatenate([[0.33], m])
    b_ext = np.concatenate([[0.0], b])
    G_ext, _ = coef.gamma_triple_sum(a_ext, m_ext, b_ext)
    np.testing.assert_allclose(G_ext[1:, 0], b_ref, rtol=1e-13)


def test_gamma_linear_recurrence_from_definition():
    """gamma_{i,j} = alpha_i gamma_{i-1,j} + beta_i prod_{u=j+1}^{i} mu_u,
    checked on the definition's own output."""
    rng = np.random.default_rng(6)
    a, m, b = _gates(rng, 12)
    G, _ = coef.gamma_triple_sum(a, m, b)
    for i in range(1, 12):
        for j in range(i):
            rhs = a[i] * G[i - 1, j] + b[i] * np.prod(m[j + 1:i + 1])
            assert abs(G[i, j] - rhs) < 1e-14


def test_chunk_vectors_shifted_entries():
    rng = np.random.default_rng(7)
    a, m, b = _gates(rng, 6)
    cv = coef.chunk_vectors(a, m, b)
    assert cv["abar_m"][0] == 1.0 and cv["b_m"][0] == 0.0
    np.testing.assert_allclose(cv["abar_m"][1:], np.cumprod(a)[:-1])
    np.testing.assert_allclose(cv["b_m"][1:], cv["b"][:-1])
    np.testing.assert_allclose(cv["mu_tail"] * cv["mubar"], cv["mubar"][-1],
                               rtol=1e-13)
    assert np.all(np.diag(cv["Gamma_m"]) == 0)
