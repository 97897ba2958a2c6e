"""GPU parity of spec_sample_rows (draft-side draws, "Accelerating Sonar
through speculation" §Target-Draft) against the oracle: the token of every
row is the oracle's inverse-CDF draw at the DRAFT-purpose uniform, except
where the oracle puts u or the top-p boundary within MARGIN of a
threshold (then the two sides may round apart); greedy is bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_parity import MARGIN

pytestmark = pytest.mark.gpu


def _gpu(x, T, top_p, seed, req, pos):
    import speculative_decoding_verification_60_gb300 as svp

    dev = torch.device("cuda:0")
    out = svp.sample_rows(x.to(dev), T, top_p, seed, torch.as_tensor(req, dtype=torch.int64).to(dev),
                          torch.as_tensor(pos, dtype=torch.int64).to(dev))
    torch.cuda.synchronize()
    return out["out_tokens"].cpu().numpy(), int(out["dev_error"].cpu()[0])


def _oracle_token(row, T, top_p, seed, req, pos):
    """(token, margin): the oracle's draw and how close it is to a rounding tie."""
    if T == 0.0:
        return oracle.argmax(row), np.inf
    p, st, tm = oracle.row_probs(row, T, top_p)
    if st != 0:
        return oracle.argmax(row), np.inf
    u = oracle.uniform(seed, int(req), int(pos), oracle.PURPOSE_DRAFT, 0)
    t, um = oracle.sample_inverse_cdf(p, u)
    return t, min(tm, um)


def _check(x, T, top_p, seed, req, pos, rows=None):
    got, err = _gpu(x, T, top_p, seed, req, pos)
    xf = x.float().numpy() if x.dtype == torch.bfloat16 else x.numpy()
    excused = 0
    for r in (range(x.shape[0]) if rows is None else rows):
        want, margin = _oracle_token(xf[r], T, top_p, seed, req[r], pos[r])
        if got[r] != want:
            assert margin < MARGIN, f"row {r}: token {got[r]} vs oracle {want} (margin {margin:.3g})"
            excused += 1
    return got, err, excused


@pytest.mark.parametrize("T,top_p", [(0.7, 1.0), (0.7, 0.9), (1.0, 0.9), (1.0, 0.5)])
def test_bf16_full_vocab(T, top_p):
    R, V = 24, 128256
    x = synth.zipf_logits(R, V, seed=31)
    rng = np.random.default_rng(1)
    req, pos = rng.integers(0, 1 << 40, R), rng.integers(0, 1 << 20, R)
    _, err, excused = _check(x, T, top_p, 123, req, pos)
    assert err == 0 and excused <= 1


@pytest.mark.parametrize("T,top_p", [(0.8, 1.0), (0.8, 0.95), (1.3, 0.6)])
def test_bf16_ragged_rows(T, top_p):
    # V odd: rows start off 16-byte boundaries (head, vectors and a tail)
    R, V = 40, 1001
    x = synth.zipf_logits(R, V, seed=32)
    req, pos = np.arange(R) + 5000, np.arange(R) * 3
    _, err, excused = _check(x, T, top_p, 9, req, pos)
    assert err == 0 and excused <= 1


@pytest.mark.parametrize("T,top_p", [(0.8, 1.0), (0.8, 0.95)])
def test_fp32_rows(T, top_p):
    R, V = 16, 4097
    x = synth.gaussian((R, V), 2.0, seed=33)
    req, pos = np.arange(R), np.full(R, 11)
    _, err, excused = _check(x, T, top_p, 4, req, pos)
    assert err == 0 and excused <= 1


def test_greedy_bit_exact():
    R, V = 8, 128256
    x = synth.zipf_logits(R, V, seed=34)
    got, err = _gpu(x, 0.0, 1.0, 0, np.arange(R), np.zeros(R))
    want = [oracle.argmax(x[r].float().numpy()) for r in range(R)]
    assert err == 0 and list(got) == want


def test_invalid_rows_and_degenerate_sizes():
    V = 300
    x = synth.gaussian((4, V), 1.0, seed=35)
    x[1, 17] = float("nan")
    x[2, 40] = float("inf")
    x[3, :] = float("-inf")
    xb = x.to(torch.bfloat16)
    req, pos = np.arange(4), np.zeros(4)
    got, err = _gpu(xb, 0.7, 0.9, 1, req, pos)
    assert err == 2  # SPEC_DEVERR_NONFINITE
    xf = xb.float().numpy()
    for r in (1, 2, 3):
        assert got[r] == oracle.argmax(xf[r]), r
    assert got[3] == 0
    # greedy on the same rows: the same argmax, no error
    got0, err0 = _gpu(xb, 0.0, 1.0, 1, req, pos)
    assert err0 == 0 and all(got0[r] == oracle.argmax(xf[r]) for r in range(4))
    # V = 1: the only token
    one, e1 = _gpu(torch.zeros(3, 1, dtype=torch.bfloat16), 0.7, 0.9, 1, np.arange(3), np.zeros(3))
    assert e1 == 0 and list(one) == [0, 0, 0]


def test_bench_size_sampled_rows_and_slot_independence():
    # the launch the bench times: 256 rows of V = 128256, T = 0.7, top-p 0.9
    R, V = 256, 128256
    x = synth.zipf_logits(R, V, seed=36)
    rng = np.random.default_rng(2)
    req, pos = rng.integers(0, 1 << 40, R), rng.integers(0, 1 << 20, R)
    rows = sorted(rng.choice(R, 64, replace=False).tolist())
    got, err, excused = _check(x, 0.7, 0.9, 55, req, pos, rows=rows)
    assert err == 0 and excused <= 1
    # a row's token depends on (row, seed, request, position), not on its slot
    sub = [3, 100, 255]
    got_sub, _ = _gpu(x[sub].contiguous(), 0.7, 0.9, 55, req[sub], pos[sub])
    assert list(got_sub) == [got[r] for r in sub]
