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
