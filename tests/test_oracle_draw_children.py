"""Pins of the oracle's tree-children draws (the draft model's top-K
candidates per node, "Accelerating Sonar through speculation" §EAGLE), which
the tree tests use to make node tokens: deterministic mode is the K largest
logits (ties by index); IID draws follow filter(softmax(x / T)), and the
first of them is the row sampler's draw; without replacement every draw is
the inverse CDF of the distribution left after the earlier draws, at round
j of the DRAFT-purpose uniform."""

import numpy as np
from scipy import stats

import oracle


def _softmax(x, T):
    z = np.exp((x - x.max()) / T)
    return z / z.sum()


def test_deterministic_children_are_the_k_largest_logits():
    x = np.array([0.5, 2.0, -1.0, 2.0, 1.5, 0.0])
    got = oracle.draw_children(x, 1.0, 1.0, 4, oracle.CHILD_DET, 0, 0, 0)
    assert list(got) == [1, 3, 4, 0]  # 2.0 at 1 and 3 (index order), then 1.5, then 0.5


def test_iid_children_follow_the_softmax_and_start_with_the_row_draw():
    rng = np.random.default_rng(8)
    x = rng.normal(0.0, 1.0, 6)
    T = 0.9
    firsts = []
    for req in range(6000):
        k = oracle.draw_children(x, T, 1.0, 3, oracle.CHILD_IID, 21, req, 4)
        firsts.extend(int(t) for t in k)
        if req < 50:
            row = oracle.sample_rows(x[None], T, 1.0, 21, [req], [4])[0]
            assert k[0] == row
    counts = np.bincount(np.array(firsts), minlength=6)
    assert stats.chisquare(counts, _softmax(x, T) * len(firsts)).pvalue > 1e-3


def test_without_replacement_is_sequential_inverse_cdf():
    rng = np.random.default_rng(9)
    x = rng.normal(0.0, 1.5, 40)
    T, seed, K = 1.1, 5, 4
    for req in range(30):
        got = oracle.draw_children(x, T, 1.0, K, oracle.CHILD_WOR, seed, req, 17)
        assert len(set(got.tolist())) == K
        p = _softmax(x, T)
        for j in range(K):
            u = oracle.uniform(seed, req, 17, oracle.PURPOSE_DRAFT, j)
            C = np.cumsum(p)
            target = u * C[-1]
            if np.min(np.abs(C - target)) < 1e-12:
                break
            want = int(np.searchsorted(C, target, side="right"))
            assert got[j] == want, (req, j)
            p = p.copy()
            p[want] = 0.0
