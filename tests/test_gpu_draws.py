"""Sampled parity at the bench's row sizes with many draws
("Accelerating Sonar through speculation", §Target-Draft; the cited rule:
accept d_i iff u_i < p(d_i)/q(d_i), then one token from norm(max(0, p - q))
at the first rejection or from p after a full accept).

A request's draws depend only on (seed, request id, position), so many
requests over full-size rows put the residual and bonus draws at many
points of their distributions.  Every request's accepted length and tokens
must be the oracle's (a mismatch is excused only where the oracle's own
decision margin is below MARGIN), and the accepted-length histogram must be
the histogram of the oracle's lengths."""

import numpy as np
import pytest
import torch

import synth
from gpu_parity import compare_linear, draft_tokens_from_oracle, oracle_linear, row_topp_margin, run_gpu_linear

pytestmark = pytest.mark.gpu


def _hist_check(got, ref, rows, k, excused):
    gh = np.bincount(got["accepted_len"][rows], minlength=k + 1)
    rh = np.bincount(ref["accepted_len"], minlength=k + 1)
    # an excused mismatch may move one request between two bins
    assert np.abs(gh - rh).sum() <= 2 * excused, (gh.tolist(), rh.tolist())


@pytest.mark.parametrize("T,top_p", [(0.7, 0.9), (1.0, 1.0), (0.6, 0.95)])
def test_many_draws_on_full_vocabulary_rows(T, top_p):
    """64 requests of k = 1 over V = 128256 bf16 rows: half the drafts are the
    draft model's own samples (accepts and residual draws), half uniform
    tokens (mostly outside q's nucleus: rejections with residual p)."""
    B, k, V, seed = 64, 1, 128256, 123
    tgt, drf = synth.linear_logits(B, k, V, "bf16", 31337)
    d = draft_tokens_from_oracle(drf, T, top_p, seed=7)
    d[B // 2:] = synth.uniform_tokens((B - B // 2, k), V, 99).numpy()
    req = np.arange(B, dtype=np.int64) * 7919 + 3
    pos = np.arange(B, dtype=np.int64) % 50 + 1
    got = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    rows = list(range(B))
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows)
    log = []
    excused = compare_linear(got, ref, rows, greedy=False, label=f"many draws T={T} p={top_p}",
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p), log=log)
    # at 128256 tokens a row's top-p boundary lies within 1e-6 of top_p in
    # mass for a few rows in a hundred; such rows may round apart
    assert excused <= B // 16, log
    _hist_check(got, ref, rows, k, excused)
    assert int(got["dev_error"][0]) == 0
    # both kinds of draw happened
    assert 0 < int((got["accepted_len"] == 0).sum()) < B


def test_bench_workload_32_requests():
    """The bench's workload (B = 256, k = 8, V = 128256, T = 0.7, top-p 0.9)
    in the launch configuration the bench times; 32 requests spread over the
    batch checked against the oracle, and their length histogram."""
    w = synth.WORKLOADS["linear-b256-k8-v128256-t0.7-p0.9"]
    B, k, V, T, top_p = w["B"], w["k"], w["V"], w["T"], w["top_p"]
    rows = list(np.linspace(0, B - 1, 32).astype(int))
    from gpu_parity import linear_case

    tgt, drf, d, req, pos, rows = linear_case(B, k, V, "bf16", T, top_p, w["data_seed"], w["seed"], device="cuda",
                                              check_rows=rows)
    got = run_gpu_linear(tgt, drf, d, T, top_p, w["seed"], req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, w["seed"], req, pos, rows)
    log = []
    excused = compare_linear(got, ref, rows, greedy=False, label="bench workload",
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p), log=log)
    assert excused <= 2, log
    _hist_check(got, ref, rows, k, excused)
    assert got["len_hist"].sum() == B
    assert np.array_equal(got["len_hist"], np.bincount(got["accepted_len"], minlength=k + 1))


@pytest.mark.parametrize("T,top_p", [(0.8, 0.9), (1.0, 1.0)])
def test_one_request_under_a_thousand_request_ids(T, top_p):
    """The rows of one request (k = 1, V = 20000) replicated under 1024
    request ids: the draws then probe the whole CDF of the request's
    residual and bonus distributions.  Every token must be the oracle's."""
    R, k, V, seed = 1024, 1, 20000, 4242
    tgt1, drf1 = synth.linear_logits(1, k, V, "bf16", 2718)
    tgt = tgt1.expand(R, k + 1, V).contiguous()
    drf = drf1.expand(R, k, V).contiguous()
    # half the requests draft a token inside both nuclei, half a uniform token
    d = np.zeros((R, k), dtype=np.int32)
    d[: R // 2] = draft_tokens_from_oracle(drf1, T, top_p, seed=3)[0]
    d[R // 2:] = synth.uniform_tokens((R - R // 2, k), V, 11).numpy()
    req = np.arange(R, dtype=np.int64) * 104729 + 17
    pos = np.full(R, 9, dtype=np.int64)
    got = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    rows = list(range(R))
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows)
    log = []
    excused = compare_linear(got, ref, rows, greedy=False, label=f"1024 ids T={T} p={top_p}",
                             margin_of=lambda b, i: row_topp_margin(tgt1, drf1, 0, i, T, top_p), log=log)
    # one row pair: its top-p margin is the same for every request
    assert excused <= 4, log
    _hist_check(got, ref, rows, k, excused)
    # the draws spread over the distributions
    t_star = got["out_tokens"][np.arange(R), got["accepted_len"]]
    assert len(np.unique(t_star)) > R // 20


def test_cut_at_the_end_of_a_region():
    """Top-p keeps the first n_keep tokens valued exactly at the boundary
    value tau, in index order.  Here the last kept one is the last
    tau-valued token of the first 1024 elements, so the tau-valued tokens
    after it are dropped everywhere after that point; 64 bonus draws over the
    row (target row 0 equals draft row 0, so every draft is accepted) must
    match the oracle and never return a dropped token."""
    V, B, k, T, seed = 8192, 64, 1, 1.0, 99
    x = np.full(V, -20.0, dtype=np.float32)
    big = [100, 2100, 3100, 4100, 5100, 6100, 7100, 8100]
    x[big] = 4.0
    taus = [10, 500, 1000, 1100, 1500, 2000, 3500, 3600, 3700]
    x[taus] = 1.0
    w = np.exp(x.astype(np.float64) - 4.0)
    top_p = float((w[big].sum() + 2.5 * w[taus[0]]) / w.sum())  # keeps exactly the first three tau-valued
    import oracle

    p = oracle.row_probs(x, T, top_p)[0]
    assert [int(p[t] > 0) for t in taus] == [1, 1, 1, 0, 0, 0, 0, 0, 0]
    g = torch.Generator().manual_seed(5)
    row0 = torch.randn(V, generator=g)
    tgt = torch.stack([row0, torch.from_numpy(x)]).unsqueeze(0).expand(B, 2, V).contiguous().to(torch.bfloat16)
    drf = row0.unsqueeze(0).unsqueeze(0).expand(B, 1, V).contiguous().to(torch.bfloat16)
    d = np.full((B, k), int(torch.argmax(row0)), dtype=np.int32)
    req = np.arange(B, dtype=np.int64) * 31 + 7
    pos = np.zeros(B, dtype=np.int64)
    got = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    assert (got["accepted_len"] == 1).all()
    dropped = set(taus[3:])
    assert not any(int(t) in dropped for t in got["out_tokens"][:, 1])
    rows = list(range(B))
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows)
    assert compare_linear(got, ref, rows, greedy=False, label="cut at a region end") == 0
    # the draws reach past the cut
    assert (got["out_tokens"][:, 1] > 1000).sum() > B // 4
