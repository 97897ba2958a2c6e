"""Pins of the oracle's per-row distributions ("Accelerating Sonar through
speculation", §Target-Draft: acceptance compares full probability
distributions) and of its inverse-CDF draw."""

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from exact_enum import ref_probs


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_matches_scipy(T):
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.normal(0, 3, 50)
        p, st, _ = oracle.row_probs(x, T, 1.0)
        assert st == 0
        np.testing.assert_allclose(p, softmax(x / T), rtol=1e-13, atol=1e-16)


@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.5, 0.8, 0.9, 0.999])
def test_top_p_matches_tie_aware_definition(top_p):
    rng = np.random.default_rng(int(top_p * 1000))
    for trial in range(40):
        V = int(rng.integers(2, 12))
        x = rng.integers(-3, 4, V).astype(np.float64) if trial % 2 else rng.normal(0, 1, V)
        T = float(rng.choice([0.5, 1.0]))
        p, st, _ = oracle.row_probs(x, T, top_p)
        assert st == 0
        np.testing.assert_allclose(p, ref_probs(x, T, top_p), rtol=1e-12, atol=1e-15)


def test_top_p_special_cases():
    x = np.array([0.0, 2.0, 2.0, 1.0, -np.inf])
    p, st, _ = oracle.row_probs(x, 1.0, 1.0)
    np.testing.assert_allclose(p[:4], softmax(x[:4]), rtol=1e-14)
    assert p[4] == 0.0
    # a tiny nucleus keeps only the top token, ties to the lower index
    p, st, _ = oracle.row_probs(x, 1.0, 1e-9)
    assert list(p) == [0.0, 1.0, 0.0, 0.0, 0.0]


def test_invalid_rows():
    for bad in ([0.0, np.nan, 1.0], [0.0, np.inf], [-np.inf, -np.inf]):
        _, st, _ = oracle.row_probs(np.array(bad), 1.0, 1.0)
        assert st == oracle.ERR_NONFINITE


def test_argmax_lowest_index_matches_numpy():
    rng = np.random.default_rng(3)
    for _ in range(50):
        x = rng.integers(-2, 3, 17).astype(np.float64)
        assert oracle.argmax(x) == int(np.argmax(x))
    assert oracle.argmax(np.array([1.0, np.inf, np.nan, 3.0, 3.0])) == 3


def test_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(4)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[0] = 1.0
        u = float(rng.integers(0, 2**24)) / 2**24
        t, _ = oracle.sample_inverse_cdf(w, u)
        assert t == int(np.searchsorted(np.cumsum(w), u * w.sum(), side="right"))
        assert w[t] > 0


def test_inverse_cdf_is_exact_on_the_uniform_grid():
    """Each token is chosen on a set of 24-bit grid points whose measure is
    its normalised weight, to one grid step."""
    rng = np.random.default_rng(5)
    for _ in range(10):
        V = 6
        w = rng.random(V)
        w[2] = 0.0
        edges = [0]
        for v in range(V):
            lo, hi = edges[-1], 2**24
            while lo < hi:  # first grid point whose draw is beyond v
                mid = (lo + hi) // 2
                if oracle.sample_inverse_cdf(w, mid / 2**24)[0] > v:
                    hi = mid
                else:
                    lo = mid + 1
            edges.append(lo)
        meas = np.diff(edges) / 2**24
        np.testing.assert_allclose(meas, w / w.sum(), atol=2.0**-23)
        assert meas[2] == 0.0


def test_zero_weights_return_minus_one():
    assert oracle.sample_inverse_cdf(np.zeros(4), 0.3)[0] == -1
