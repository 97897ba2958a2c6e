"""Pins of the oracle's linear verification ("Accelerating Sonar through
speculation", §Speculative decoding and §Target-Draft; rule of the cited
"Fast Inference from Transformers via Speculative Decoding")."""

import numpy as np
import pytest
from scipy.stats import chisquare

import oracle
from exact_enum import ToyWorld, linear_emitted_distribution, max_abs_diff, ref_probs


@pytest.mark.parametrize("V,k,T,top_p", [(3, 1, 1.0, 1.0), (3, 2, 1.0, 1.0), (4, 3, 0.7, 1.0),
                                         (4, 2, 1.0, 0.8), (5, 2, 0.6, 0.7)])
def test_emitted_distribution_equals_target_exactly(V, k, T, top_p):
    w = ToyWorld(V, k, seed=100 * V + 10 * k + int(10 * top_p), T=T, top_p=top_p)
    dist = linear_emitted_distribution(w, k)
    ref = w.target_joint(k + 1)
    assert max_abs_diff(dist, ref) < 1e-12


def test_emitted_distribution_with_ties_and_top_p():
    w = ToyWorld(4, 2, seed=9, T=1.0, top_p=0.75, integer_logits=True)
    assert max_abs_diff(linear_emitted_distribution(w, 2), w.target_joint(3)) < 1e-12


def _batch_from_world(w, k, R, seed):
    """R independent requests whose drafts are drawn from the toy draft
    model with the oracle's Philox draft draws."""
    V = w.V
    tgt = np.zeros((R, k + 1, V))
    drf = np.zeros((R, k, V))
    d = np.zeros((R, k), dtype=np.int32)
    for r in range(R):
        pre = ()
        for i in range(k):
            tgt[r, i] = w.P[pre]
            drf[r, i] = w.Q[pre]
            d[r, i] = oracle.sample_rows(drf[r, i][None], w.T, w.top_p, seed, [r], [1000 + i])[0]
            pre = pre + (int(d[r, i]),)
        tgt[r, k] = w.P[pre]
    return tgt, drf, d


def test_philox_driven_batch_matches_target_chi_square():
    k, R = 2, 6000
    w = ToyWorld(3, k, seed=77, T=1.0, top_p=1.0)
    tgt, drf, d = _batch_from_world(w, k, R, seed=5)
    out = oracle.verify_linear(tgt, drf, d, w.T, w.top_p, seed=123, positions=np.full(R, 10))
    rng = np.random.default_rng(0)
    counts = {}
    for r in range(R):
        a = out["accepted_len"][r]
        seq = [int(t) for t in out["out_tokens"][r, :a + 1]]
        while len(seq) < k + 1:
            seq.append(int(rng.choice(w.V, p=w.p(tuple(seq)))))
        counts[tuple(seq)] = counts.get(tuple(seq), 0) + 1
    ref = w.target_joint(k + 1)
    keys = sorted(ref)
    obs = np.array([counts.get(s, 0) for s in keys], dtype=float)
    exp = np.array([ref[s] for s in keys]) * R
    assert chisquare(obs, exp).pvalue > 1e-4


def test_expected_accepted_length_closed_form():
    """E[a | d] = sum_j prod_{i<=j} min(1, p_i/q_i); Monte Carlo over seeds
    must agree within 4 sigma."""
    rng = np.random.default_rng(8)
    k, V = 4, 6
    tgt = rng.normal(0, 1, (1, k + 1, V))
    drf = tgt[:, :k] + rng.normal(0, 0.6, (1, k, V))
    d = np.array([[1, 3, 0, 2]], dtype=np.int32)
    r = np.array([ref_probs(tgt[0, i], 1.0, 1.0)[d[0, i]] / ref_probs(drf[0, i], 1.0, 1.0)[d[0, i]]
                  for i in range(k)])
    c = np.minimum(1.0, r)
    expect = sum(np.prod(c[:j + 1]) for j in range(k))
    n = 4000
    tb = np.repeat(tgt, n, 0)
    db = np.repeat(drf, n, 0)
    dd = np.repeat(d, n, 0)
    out = oracle.verify_linear(tb, db, dd, 1.0, 1.0, seed=99, req_ids=np.arange(n) * 7919)
    a = out["accepted_len"].astype(float)
    assert abs(a.mean() - expect) < 4 * a.std() / np.sqrt(n) + 1e-12


def test_alpha_identity_on_residual():
    """sum_v max(0, p - q) = 1 - sum_v min(p, q) (total-variation identity)."""
    rng = np.random.default_rng(9)
    for _ in range(20):
        V, k = 7, 1
        tgt = rng.normal(0, 1, (k + 1, V))
        drf = rng.normal(0, 1, (k, V))
        out = oracle.linear_request(tgt, drf, np.array([2]), 1.0, 1.0, [1.0 - 2**-53], [0.3], 0.3,
                                    want_trace=True)
        if out["trace"]["final_kind"] != 0:
            continue
        p, q = ref_probs(tgt[0], 1.0, 1.0), ref_probs(drf[0], 1.0, 1.0)
        assert abs(out["trace"]["final_w"].sum() - (1.0 - np.minimum(p, q).sum())) < 1e-14


def test_bound_n_plus_one_and_padding():
    rng = np.random.default_rng(10)
    B, k, V = 64, 5, 9
    tgt = rng.normal(0, 1, (B, k + 1, V))
    drf = tgt[:, :k] + rng.normal(0, 0.5, (B, k, V))
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    for T, tp in ((1.0, 1.0), (0.8, 0.9), (0.0, 1.0)):
        out = oracle.verify_linear(tgt, drf if T else None, d, T, tp, seed=1)
        for b in range(B):
            a = out["accepted_len"][b]
            assert 0 <= a <= k
            row = out["out_tokens"][b]
            assert list(row[:a]) == list(d[b, :a])
            assert 0 <= row[a] < V
            assert np.all(row[a + 1:] == -1)
        assert out["len_hist"].sum() == B


def test_greedy_is_argmax_comparison():
    rng = np.random.default_rng(11)
    B, k, V = 50, 4, 8
    tgt = rng.integers(-2, 3, (B, k + 1, V)).astype(np.float64)
    g = np.argmax(tgt, axis=-1)
    d = np.where(rng.random((B, k)) < 0.7, g[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    out = oracle.verify_linear(tgt, None, d, 0.0, 1.0, seed=0)
    for b in range(B):
        a = 0
        while a < k and d[b, a] == g[b, a]:
            a += 1
        assert out["accepted_len"][b] == a
        assert out["out_tokens"][b, a] == g[b, a]


def test_tiny_temperature_equals_greedy():
    """With T -> 0 and drafts taken greedily from the draft model (q one-hot
    at d), sampled verification reduces to the argmax comparison."""
    rng = np.random.default_rng(12)
    B, k, V = 30, 3, 10
    tgt = rng.normal(0, 1, (B, k + 1, V))
    drf = tgt[:, :k] + rng.normal(0, 0.5, (B, k, V))
    d = np.argmax(drf, axis=-1).astype(np.int32)
    s = oracle.verify_linear(tgt, drf, d, 1e-4, 1.0, seed=4)
    gr = oracle.verify_linear(tgt, None, d, 0.0, 1.0, seed=4)
    assert 0 < gr["accepted_len"].sum() < B * k
    assert np.array_equal(s["accepted_len"], gr["accepted_len"])
    assert np.array_equal(s["out_tokens"], gr["out_tokens"])


def test_identical_models_accept_everything():
    rng = np.random.default_rng(13)
    B, k, V = 20, 6, 12
    tgt = rng.normal(0, 1, (B, k + 1, V))
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    out = oracle.verify_linear(tgt, tgt[:, :k].copy(), d, 0.9, 1.0, seed=2)
    assert np.all(out["accepted_len"] == k)


def test_one_hot_draft_on_zero_target_rejects():
    V, k = 6, 2
    tgt = np.zeros((1, k + 1, V))
    tgt[0, 0, 3] = -np.inf
    drf = np.full((1, k, V), -np.inf)
    drf[0, :, 3] = 0.0
    out = oracle.verify_linear(tgt, drf, np.array([[3, 3]]), 1.0, 1.0, seed=3)
    assert out["accepted_len"][0] == 0
    assert out["out_tokens"][0, 0] != 3


def test_invalid_inputs_fall_back():
    rng = np.random.default_rng(14)
    B, k, V = 3, 2, 5
    tgt = rng.normal(0, 1, (B, k + 1, V))
    drf = rng.normal(0, 1, (B, k, V))
    d = np.array([[0, 1], [7, 1], [2, 2]], dtype=np.int32)
    tgt[2, 1, 4] = np.nan
    out = oracle.verify_linear(tgt, drf, d, 1.0, 1.0, seed=3)
    assert out["dev_error"] == oracle.ERR_TOKEN | oracle.ERR_NONFINITE
    for b in (1, 2):
        assert out["accepted_len"][b] == 0
        assert out["out_tokens"][b, 0] == np.argmax(tgt[b, 0])
