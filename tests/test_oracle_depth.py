"""Pins of the oracle's per-depth acceptance statistics ("M7.8 - Speculative Serving", sections
0x02D "Estimation Bias And Censoring" and 0x07B): alpha_hat_j = n_accepted_j / n_reached_j and
E[A] = sum_{j<=gamma} prod_{m<=j} alpha_hat_m, against exact fractions, the constant-alpha closed
form of SOTA-227 ("Why it is free rather than a trade"), and a simulation with known rates."""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _row_off(K):
    return np.concatenate([[0], np.cumsum(np.asarray(K) + 1)]).astype(np.int32)


def test_hand_example_with_a_bad_request():
    # four requests with K = 3; A = 0, 1, 3; the fourth has a status bit and does not count
    K = [3, 3, 3, 3]
    A = np.array([0, 1, 3, 2], np.int32)
    status = np.array([0, 0, 0, 1], np.int32)
    nr, na = oracle.depth_counts(_row_off(K), A, status, 4)
    assert nr.tolist() == [3, 2, 1, 0]    # depth 2 needs A >= 1, depth 3 A >= 2, depth 4 K >= 4
    assert na.tolist() == [2, 1, 1, 0]
    ah = [Fraction(2, 3), Fraction(1, 2), Fraction(1, 1)]
    pooled = Fraction(2 + 1 + 1, 3 + 2 + 1)
    got = oracle.depth_alpha(nr, na, 0.25, 6)
    want = ah + [pooled] * 3                # depth 4 was reached by nobody: the pooled rate
    assert np.allclose(got, [float(x) for x in want], rtol=0, atol=1e-15)
    for g in range(0, 7):
        ea, prod = Fraction(0), Fraction(1)
        for j in range(g):
            prod *= want[j]
            ea += prod
        assert oracle.depth_expected_accept(nr, na, 0.25, g) == pytest.approx(float(ea), abs=1e-14)
        c = Fraction(1, 10)
        f = (1 + ea) / (g * c + 1)
        assert oracle.depth_objective(nr, na, 0.25, 0.1, g) == pytest.approx(float(f), abs=1e-14)


def test_nothing_reached_keeps_the_previous_estimate():
    nr = np.zeros(5, np.int32)
    na = np.zeros(5, np.int32)
    assert np.allclose(oracle.depth_alpha(nr, na, 0.6, 5), 0.6)
    g, ea = oracle.choose_gamma_depth(nr, na, 0.6, 0.05, 0, 8)
    g0, _ = oracle.choose_gamma(0.0, 0, 0.6, 0.05, 0, 8)
    assert g == g0


@pytest.mark.parametrize("alpha,c", [(Fraction(1, 2), 0.05), (Fraction(3, 4), 0.1), (Fraction(7, 8), 0.02)])
def test_constant_rates_reduce_to_the_closed_form(alpha, c):
    # counts with the same rate at every depth: alpha_hat_j = alpha exactly
    n0 = 8 ** 4
    nr = np.array([n0 * alpha ** j for j in range(4)], np.float64)
    na = nr * float(alpha)
    assert np.all(nr == np.round(nr)) and np.all(na == np.round(na))
    nr, na = nr.astype(np.int32), na.astype(np.int32)
    for g in range(0, 10):
        assert oracle.depth_objective(nr, na, 0.0, c, g) == pytest.approx(
            oracle.gamma_objective(float(alpha), c, g), rel=1e-13)
    g_depth, ea = oracle.choose_gamma_depth(nr, na, 0.0, c, 0, 9)
    g_const, a = oracle.choose_gamma(float(alpha), 1, 0.0, c, 0, 9)
    assert g_depth == g_const
    assert ea == pytest.approx(float(sum(alpha ** j for j in range(1, g_depth + 1))), rel=1e-13)


def test_censoring_differs_from_the_naive_rate():
    # the naive estimator n_accepted_j / n_rounds understates deeper positions
    K = [4] * 6
    A = np.array([4, 4, 2, 0, 1, 3], np.int32)
    nr, na = oracle.depth_counts(_row_off(K), A, np.zeros(6, np.int32), 4)
    naive = na / 6.0
    hat = na / nr
    assert nr.tolist() == [6, 5, 4, 3] and na.tolist() == [5, 4, 3, 2]
    assert np.all(hat[1:] > naive[1:])


def test_simulated_rates_are_recovered():
    # Bernoulli acceptance with known per-depth rates; A = leading successes
    rng = np.random.default_rng(4)
    rates = np.array([0.9, 0.7, 0.5, 0.3, 0.8])
    Kmax, n = len(rates), 40000
    K = rng.integers(0, Kmax + 1, size=n)
    succ = rng.random((n, Kmax)) < rates
    A = np.zeros(n, np.int32)
    for i in range(n):
        a = 0
        while a < K[i] and succ[i, a]:
            a += 1
        A[i] = a
    nr, na = oracle.depth_counts(_row_off(K), A, np.zeros(n, np.int32), Kmax)
    hat = na / nr
    sd = np.sqrt(rates * (1 - rates) / nr)
    assert np.all(np.abs(hat - rates) < 4 * sd), (hat, rates, sd)
