"""Pins of the oracle's row sampler, the draft model's own draws
("Accelerating Sonar through speculation", §Target-Draft): the draws follow
filter(softmax(x / T)) written out here from its definition, the top-p
nucleus is respected, greedy is the lowest-index maximum, and each draw is
the inverse CDF at the DRAFT-purpose uniform of its (request, position)."""

import numpy as np
from scipy import stats

import oracle


def _softmax(x, T):
    z = np.exp((x - x.max()) / T)
    return z / z.sum()


def _draws(x, T, top_p, n, seed=3):
    """n draws from the one row x, each with its own request id."""
    X = np.ascontiguousarray(np.broadcast_to(np.asarray(x, dtype=np.float64), (n, len(x))))
    return oracle.sample_rows(X, T, top_p, seed, req=np.arange(n), pos=np.full(n, 7))


def _chi2_pvalue(tokens, p):
    keep = p > 0
    counts = np.bincount(tokens, minlength=p.size)
    assert counts[~keep].sum() == 0, "a token outside the support was drawn"
    return stats.chisquare(counts[keep], p[keep] * len(tokens)).pvalue


def test_draws_follow_softmax():
    x = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -3.0])
    T = 0.8
    t = _draws(x, T, 1.0, 20000)
    assert _chi2_pvalue(t, _softmax(x, T)) > 1e-3


def test_draws_follow_the_nucleus():
    # probabilities 0.5, 0.3, 0.1, 0.05, 0.03, 0.02 at T = 1: the smallest
    # prefix (by descending probability) reaching 0.85 is {0, 1, 2}
    p = np.array([0.5, 0.3, 0.1, 0.05, 0.03, 0.02])
    x = np.log(p)
    t = _draws(x, 1.0, 0.85, 20000)
    q = np.where(np.arange(6) < 3, p, 0.0)
    assert _chi2_pvalue(t, q / q.sum()) > 1e-3
    # a temperature flattens the row before the filter: at T = 2 the
    # probabilities are proportional to sqrt(p) and the nucleus grows
    s = np.sqrt(p) / np.sqrt(p).sum()
    order = np.argsort(-s, kind="stable")
    before = np.concatenate([[0.0], np.cumsum(s[order])[:-1]])
    kept = order[before < 0.85]
    q2 = np.zeros(6)
    q2[kept] = s[kept]
    t2 = _draws(x, 2.0, 0.85, 20000, seed=4)
    assert _chi2_pvalue(t2, q2 / q2.sum()) > 1e-3


def test_greedy_is_lowest_index_max_over_finite_entries():
    x = np.array([[1.0, 3.0, np.nan, 3.0, np.inf, -1.0]])
    assert oracle.sample_rows(x, 0.0, 1.0, 0, [0], [0])[0] == 1
    # a sampled row with a NaN or +inf falls back to the same argmax
    assert oracle.sample_rows(x, 0.7, 0.9, 0, [0], [0])[0] == 1
    # no entry other than NaN / +inf: token 0
    y = np.array([[np.nan, np.inf, np.nan]])
    assert oracle.sample_rows(y, 0.0, 1.0, 0, [0], [0])[0] == 0


def test_each_draw_is_the_inverse_cdf_at_the_draft_uniform():
    rng = np.random.default_rng(5)
    x = rng.normal(0.0, 2.0, 100)
    T, seed = 0.9, 77
    C = np.cumsum(_softmax(x, T))
    checked = 0
    for req in range(40):
        pos = int(rng.integers(0, 1 << 40))
        u = oracle.uniform(seed, req, pos, oracle.PURPOSE_DRAFT, 0)
        target = u * C[-1]
        want = int(np.searchsorted(C, target, side="right"))  # smallest v with C(v) > u * C(V-1)
        if np.min(np.abs(C - target)) < 1e-12:
            continue
        got = oracle.sample_rows(x[None], T, 1.0, seed, [req], [pos])[0]
        assert got == want, (req, pos)
        checked += 1
    assert checked >= 35
    # the purpose is part of the counter: the DRAFT uniforms are not the BONUS ones
    others = [oracle.uniform(seed, r, 9, oracle.PURPOSE_BONUS, 0) for r in range(20)]
    drafts = [oracle.uniform(seed, r, 9, oracle.PURPOSE_DRAFT, 0) for r in range(20)]
    assert others != drafts
