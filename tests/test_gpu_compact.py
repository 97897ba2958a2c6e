"""GPU parity of spec_compact_accepted against the oracle, bit for bit
("Accelerating Sonar through speculation", §MTP and §MTP schedule for a
single token)."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_parity import spec_bits

pytestmark = pytest.mark.gpu


def _run(hid, acc, ot, path=None):
    import speculative_decoding_verification_60_gb300 as svp

    dev = torch.device("cuda:0")
    out = svp.compact_accepted(hid.to(dev), torch.as_tensor(acc, dtype=torch.int32).to(dev),
                               torch.as_tensor(ot, dtype=torch.int32).to(dev),
                               None if path is None else torch.as_tensor(path, dtype=torch.int32).to(dev))
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


def _check(hid, acc, ot, path=None):
    got = _run(hid, acc, ot, path)
    bits = hid.contiguous().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.compact(bits, acc, ot, path)
    n = int(ref["offsets"][-1])
    assert got["offsets"].numpy().tolist() == ref["offsets"].tolist()
    assert np.array_equal(got["next_tokens"].numpy()[:n], ref["next_tokens"])
    g = got["out_hidden"][:n].contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(g, ref["out_hidden"])
    assert int(got["dev_error"][0]) == spec_bits(ref["dev_error"])


def test_golden_fixture():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "compact_mtp_shift.json")))
    B, T, H = g["B"], g["T"], g["H"]
    hid = np.zeros((B, T, H), dtype=np.uint16)
    for b in range(B):
        for r in range(T):
            hid[b, r] = [100 * b + 10 * r, 100 * b + 10 * r + 1]
    h = torch.from_numpy(hid.view(np.int16)).view(torch.bfloat16)
    got = _run(h, g["accepted_len"], g["out_tokens"])
    assert got["offsets"].tolist() == g["expect_offsets"]
    assert got["next_tokens"][:7].tolist() == g["expect_next_tokens"]
    assert got["out_hidden"][:7].view(torch.int16).numpy().view(np.uint16).tolist() == g["expect_rows"]
    got = _run(h, g["accepted_len"], g["out_tokens"], g["tree_path_nodes"])
    assert got["out_hidden"][:7].view(torch.int16).numpy().view(np.uint16).tolist() == g["expect_tree_rows"]


@pytest.mark.parametrize("B,T,H", [(5, 4, 8), (37, 4, 7168), (9, 6, 1001), (1, 1, 3)])
def test_random_cases(B, T, H):
    rng = np.random.default_rng(B * 100 + H)
    hid = synth.hidden_states(B, T, H, seed=B + H)
    W = T
    acc = rng.integers(0, W, B).astype(np.int32)
    ot = rng.integers(0, 5000, (B, W)).astype(np.int32)
    _check(hid, acc, ot)
    path = np.stack([rng.permutation(T)[:W] for _ in range(B)]).astype(np.int32)
    _check(hid, acc, ot, path)


def test_full_size_workload_from_verification():
    import speculative_decoding_verification_60_gb300 as svp

    w = synth.WORKLOADS["linear-b1024-k3-v129280-h7168"]
    B, k, V, H = w["B"], w["k"], w["V"], w["H"]
    tgt, drf = synth.linear_logits(B, k, V, "bf16", w["data_seed"], device="cuda")
    d = torch.argmax(drf.float(), dim=-1).to(torch.int32)
    out = svp.verify_linear(tgt, drf, d, 1.0, 1.0, w["seed"])
    hid = synth.hidden_states(B, k + 1, H, seed=w["data_seed"], device="cuda")
    acc = out["accepted_len"].cpu().numpy()
    ot = out["out_tokens"].cpu().numpy()
    _check(hid.cpu(), acc, ot)


def test_bad_lengths_are_flagged():
    hid = synth.hidden_states(3, 4, 16, seed=1)
    acc = np.array([1, 7, -2], dtype=np.int32)
    ot = np.arange(12, dtype=np.int32).reshape(3, 4)
    _check(hid, acc, ot)
    path = np.array([[0, 9, -1, -1], [0, 1, 2, 3], [0, 1, 2, 3]], dtype=np.int32)
    _check(hid, np.array([1, 0, 2], dtype=np.int32), ot, path)
