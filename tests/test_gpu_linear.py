"""GPU parity of spec_verify_linear against the oracle, through the C ABI
("Accelerating Sonar through speculation", §Speculative decoding and
§Target-Draft)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_parity import compare_linear, linear_case, oracle_linear, row_topp_margin, run_gpu_linear, spec_bits

pytestmark = pytest.mark.gpu

SMALL = [
    # B, k, V, dtype, T, top_p
    (1, 4, 32, "f32", 1.0, 1.0),      # the tiny fp32 workload
    (64, 4, 32, "f32", 1.0, 1.0),
    (64, 4, 32, "f32", 0.0, 1.0),
    (16, 3, 1000, "bf16", 1.0, 1.0),
    (16, 3, 1000, "bf16", 0.7, 0.9),
    (12, 2, 1001, "bf16", 0.7, 0.9),   # rows not 16-byte aligned
    (12, 2, 1001, "bf16", 0.0, 1.0),
    (6, 4, 20011, "bf16", 1.0, 0.8),   # several tiles and a ragged tail
    (6, 4, 20011, "bf16", 1.3, 1.0),
    (8, 3, 5003, "f32", 0.9, 0.9),     # fp32 nucleus by key bisection
    (8, 1, 7, "bf16", 1.0, 0.5),       # shorter than one vector
    (4, 8, 65536 + 17, "bf16", 0.7, 0.9),
]


@pytest.mark.parametrize("B,k,V,dtype,T,top_p", SMALL)
def test_small_cases_match_oracle(B, k, V, dtype, T, top_p):
    seed = 42
    tgt, drf, d, req, pos, rows = linear_case(B, k, V, dtype, T, top_p, data_seed=1000 + V + k, seed=seed)
    got = run_gpu_linear(tgt, drf if T > 0 else None, d, T, top_p, seed, req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows)
    excused = compare_linear(got, ref, rows, greedy=(T == 0.0), label=f"V={V}",
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))
    assert excused <= max(1, B // 50)
    assert np.array_equal(got["len_hist"], np.bincount(got["accepted_len"], minlength=k + 1))
    assert int(got["dev_error"][0]) == 0


@pytest.mark.parametrize("name,T,top_p,check", [
    ("linear-b64-k4-v128256", 1.0, 1.0, 8),
    ("linear-b256-k8-v128256-t0.7-p0.9", 0.7, 0.9, 6),
    ("linear-b1024-k3-v129280-h7168", 1.0, 1.0, 8),
    ("linear-b1024-k3-v129280-h7168", 0.0, 1.0, None),
    ("linear-b256-k8-v128256-t0.7-p0.9", 0.0, 1.0, None),
])
def test_full_size_workloads(name, T, top_p, check):
    w = synth.WORKLOADS[name]
    B, k, V = w["B"], w["k"], w["V"]
    dev = "cuda"
    rows = None if check is None else list(np.linspace(0, B - 1, check).astype(int))
    tgt, drf, d, req, pos, rows = linear_case(B, k, V, "bf16", T, top_p, w["data_seed"], w["seed"], device=dev,
                                              check_rows=rows)
    got = run_gpu_linear(tgt, drf if T > 0 else None, d, T, top_p, w["seed"], req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, w["seed"], req, pos, rows)
    excused = compare_linear(got, ref, rows, greedy=(T == 0.0), label=name,
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))
    assert excused <= 1
    assert got["len_hist"].sum() == B


@pytest.mark.parametrize("V", [3000, 3001])
def test_results_do_not_depend_on_batch_slot(V):
    """Bit for bit when rows are 16-byte aligned (V a multiple of 8); with an
    odd V the slot changes the summation order, so only margin cases may
    differ."""
    B, k, T, top_p, seed = 24, 4, 0.8, 0.95, 9
    tgt, drf, d, req, pos, rows = linear_case(B, k, V, "bf16", T, top_p, data_seed=77, seed=seed)
    full = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    sel = [17, 3, 9]
    part = run_gpu_linear(tgt[sel], drf[sel], d[sel], T, top_p, seed, req[sel], pos[sel])
    if V % 8 == 0:
        for j, b in enumerate(sel):
            assert full["accepted_len"][b] == part["accepted_len"][j]
            assert np.array_equal(full["out_tokens"][b], part["out_tokens"][j])
            assert np.array_equal(full["token_probs"][b], part["token_probs"][j])
    else:
        ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, sel)
        mg = lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p)  # noqa: E731
        compare_linear(full, ref, sel, greedy=False, label="full batch", margin_of=mg)
        sub = {key: v for key, v in part.items()}
        compare_linear(sub, ref, range(len(sel)), greedy=False, label="sub batch",
                       margin_of=lambda j, i: row_topp_margin(tgt, drf, sel[j], i, T, top_p))


def test_repeatable_bit_for_bit():
    B, k, V, T, top_p, seed = 16, 5, 9000, 0.7, 0.9, 3
    tgt, drf, d, req, pos, rows = linear_case(B, k, V, "bf16", T, top_p, data_seed=78, seed=seed)
    a = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    b = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    for key in ("accepted_len", "out_tokens", "accept_prob", "token_probs"):
        assert np.array_equal(a[key], b[key]), key


def test_invalid_inputs_take_the_defined_fallback():
    B, k, V, T, top_p, seed = 6, 3, 600, 1.0, 0.9, 1
    tgt, drf, d, req, pos, rows = linear_case(B, k, V, "bf16", T, top_p, data_seed=79, seed=seed)
    tgt = tgt.clone()
    drf = drf.clone()
    d[1, 2] = V + 5                        # token out of range
    tgt[2, 1, 17] = float("nan")           # NaN in a target row
    drf[3, 0, 4] = float("inf")            # +inf in a draft row
    tgt[4, :, : V // 2] = float("-inf")    # a masked half: allowed, zero probability
    got = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows)
    assert int(got["dev_error"][0]) == spec_bits(oracle.ERR_TOKEN | oracle.ERR_NONFINITE)
    assert int(got["dev_error"][0]) == spec_bits(ref["dev_error"])
    compare_linear(got, ref, rows, greedy=False, label="invalid",
                   margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))
    for b in (1, 2, 3):
        assert got["accepted_len"][b] == 0
        assert got["out_tokens"][b, 0] == oracle.argmax(tgt[b, 0])


def test_ties_and_constant_rows():
    B, k, V = 8, 3, 2048
    g = torch.Generator().manual_seed(5)
    tgt = torch.randint(-3, 4, (B, k + 1, V), generator=g).to(torch.bfloat16)
    drf = torch.randint(-3, 4, (B, k, V), generator=g).to(torch.bfloat16)
    tgt[0] = 0.0                            # every logit equal
    drf[0] = 0.0
    tgt[1, :, 5] = 100.0                    # one dominant token, duplicated below
    tgt[1, :, 900] = 100.0
    req = np.arange(B, dtype=np.int64)
    pos = np.zeros(B, dtype=np.int64)
    for T, top_p in ((0.0, 1.0), (1.0, 1.0), (0.5, 0.7), (2.0, 0.3)):
        d = np.zeros((B, k), dtype=np.int32)
        for b in range(B):
            d[b] = oracle.sample_rows(drf[b], T if T > 0 else 1.0, top_p, seed=2, req=np.full(k, b), pos=np.arange(k))
        got = run_gpu_linear(tgt, drf if T > 0 else None, d, T, top_p, 11, req, pos)
        ref = oracle_linear(tgt, drf, d, T, top_p, 11, req, pos, range(B))
        compare_linear(got, ref, range(B), greedy=(T == 0.0), label=f"ties T={T} p={top_p}",
                       margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))


@pytest.mark.parametrize("gap", [1.0, -1.0])
def test_far_tail_draft_token_decides_like_the_oracle(gap):
    """Caller-supplied drafts in the far tail of q: q(d) underflows in fp32
    (about e^-250 of the row maximum) while p(d) / q(d) stays moderate (e^gap
    times the normalisers' ratio).  The decision must follow the exact
    ratio, as the fp64 oracle takes it ("Fast Inference from Transformers
    via Speculative Decoding": accept with probability min(1, p/q))."""
    B, k, V, T, top_p, seed = 8, 2, 256, 1.0, 1.0, 3
    g = torch.Generator().manual_seed(41)
    tgt = torch.randn(B, k + 1, V, generator=g)
    drf = tgt[:, :k] + 0.3 * torch.randn(B, k, V, generator=g)
    d = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        for i in range(k):
            x = (b * 37 + i * 11) % V
            d[b, i] = x
            drf[b, i, x] = -250.0
            tgt[b, i, x] = -250.0 + gap
    tgt, drf = tgt.to(torch.bfloat16), drf.to(torch.bfloat16)
    req = np.arange(B, dtype=np.int64) + 5
    pos = np.arange(B, dtype=np.int64) * 2
    got = run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos)
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, range(B))
    assert np.array_equal(got["accepted_len"], ref["accepted_len"])
    assert np.array_equal(got["out_tokens"], ref["out_tokens"])
    np.testing.assert_allclose(got["accept_prob"], ref["accept_prob"], rtol=1e-5, atol=1e-6)
    if gap > 0:  # p/q > 1 on every drafted token: everything accepted
        assert np.all(got["accepted_len"] == k)
    assert int(got["dev_error"][0]) == 0
