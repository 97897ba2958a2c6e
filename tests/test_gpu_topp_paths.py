"""GPU parity of the exact top-p nucleus on rows built to send the row
statistics down each of its routes: a bracket entirely below zero, a
bracket spanning zero (values within 2^-10 of zero measured as one lump), a
boundary inside that lump (counted key by key), and peaked rows.  The
probabilities must match the oracle's ("Accelerating Sonar through
speculation", §Target-Draft: full distributions compared; top-p on p and q
alike)."""

import numpy as np
import pytest
import torch

import oracle
from gpu_parity import PROB_TOL, compare_linear, draft_tokens_from_oracle, oracle_linear, row_topp_margin, run_gpu_linear

pytestmark = pytest.mark.gpu


def _rows(kind: str, B: int, k: int, V: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    n = B * (2 * k + 1)
    if kind == "gauss":  # plain N(0,1): at T=1 the boundary of top-p 0.9 sits near -0.28
        x = torch.randn(n, V, generator=g)
    elif kind == "tiny":  # most of the mass within 2^-11 of zero, a few larger values
        x = (torch.rand(n, V, generator=g) * 2 - 1) * 2.0 ** -11
        x[:, :8] = torch.randn(n, 8, generator=g) * 0.5
    elif kind == "peaked":  # one dominant token per row over N(0,1)
        x = torch.randn(n, V, generator=g)
        x[torch.arange(n), torch.randint(0, V, (n,), generator=g)] += 14.0
    else:
        raise ValueError(kind)
    x = x.to(torch.bfloat16)
    tgt = x[: B * (k + 1)].reshape(B, k + 1, V).contiguous()
    drf = x[B * (k + 1):].reshape(B, k, V).contiguous()
    return tgt, drf


@pytest.mark.parametrize("kind,T,top_p", [
    ("gauss", 1.0, 0.9),     # bracket below zero
    ("gauss", 1.0, 0.841),   # boundary near zero: the bracket spans it
    ("gauss", 0.5, 0.97),
    ("tiny", 1.0, 0.5),      # boundary inside the near-zero lump
    ("tiny", 1.0, 0.97),
    ("peaked", 0.7, 0.9),    # boundary at the dominant token
    ("peaked", 1.0, 0.999),
])
def test_topp_routes_match_oracle(kind, T, top_p):
    B, k, V, seed = 6, 2, 6000, 21
    tgt, drf = _rows(kind, B, k, V, seed={"gauss": 11, "tiny": 12, "peaked": 13}[kind] * 1000 + int(top_p * 1000))
    d = draft_tokens_from_oracle(drf, T, top_p, seed=3)
    req = np.arange(B, dtype=np.int64) + 40
    pos = np.arange(B, dtype=np.int64) * 3
    got = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, range(B))
    excused = compare_linear(got, ref, range(B), greedy=False, label=f"{kind} T={T} p={top_p}",
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))
    assert excused <= 1
    assert int(got["dev_error"][0]) == 0


def test_lump_rows_token_probabilities_are_exact():
    """Every drafted token probability of rows whose boundary lies within
    2^-10 of zero, against the oracle's filtered row."""
    B, k, V, T, top_p = 4, 3, 4096, 1.0, 0.6
    tgt, drf = _rows("tiny", B, k, V, seed=5)
    d = draft_tokens_from_oracle(drf, T, top_p, seed=9)
    got = run_gpu_linear(tgt, drf, d, T, top_p, 1, np.arange(B), np.zeros(B, dtype=np.int64))
    for b in range(B):
        for i in range(k):
            p = oracle.row_probs(tgt[b, i], T, top_p)[0]
            q = oracle.row_probs(drf[b, i], T, top_p)[0]
            tok = int(d[b, i])
            if row_topp_margin(tgt, drf, b, i, T, top_p) < 1e-6:
                continue
            assert abs(float(got["token_probs"][b, i, 0]) - p[tok]) < PROB_TOL
            assert abs(float(got["token_probs"][b, i, 1]) - q[tok]) < PROB_TOL


@pytest.mark.parametrize("shift", [-3.0, 3.0])
def test_misleading_layout_still_exact(shift):
    """Rows whose values depend on the position modulo 8 and modulo 16384,
    so that any fixed-stride sample of the row sees a shifted distribution;
    whatever bracket an estimate picks, the result must stay exact."""
    B, k, V, T, top_p = 4, 2, 40000, 1.0, 0.9
    g = torch.Generator().manual_seed(77)
    n = B * (2 * k + 1)
    x = torch.randn(n, V, generator=g)
    idx = torch.arange(V)
    odd = ((idx % 8) % 4 == 0) & ((idx % 16384) < 4096)
    x[:, odd] += shift
    x = x.to(torch.bfloat16)
    tgt = x[: B * (k + 1)].reshape(B, k + 1, V).contiguous()
    drf = x[B * (k + 1):].reshape(B, k, V).contiguous()
    d = draft_tokens_from_oracle(drf, T, top_p, seed=4)
    req = np.arange(B, dtype=np.int64)
    pos = np.zeros(B, dtype=np.int64)
    got = run_gpu_linear(tgt, drf, d, T, top_p, 8, req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, 8, req, pos, range(B))
    excused = compare_linear(got, ref, range(B), greedy=False, label=f"layout shift {shift}",
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))
    assert excused <= 1
