"""GPU parity of spec_verify_linear_compact: linear verification and the
compaction of the accepted positions in the same launches ("Accelerating
Sonar through speculation", §MTP: token t_{i+1} pairs with hidden state
H_i; §MTP schedule for a single token: a kernel inserts the next target
tokens).  The verification outputs must be those of spec_verify_linear,
the compaction those of the oracle's compaction of them, bit for bit."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_parity import compare_linear, linear_case, oracle_linear, row_topp_margin

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _fused(tgt, drf, d, hid, T, top_p, seed, req=None, pos=None):
    import speculative_decoding_verification_60_gb300 as svp

    out = svp.verify_linear_compact(tgt.to(DEV), None if drf is None else drf.to(DEV),
                                    torch.as_tensor(d, dtype=torch.int32).to(DEV), hid.to(DEV), T, top_p, seed,
                                    request_ids=None if req is None else torch.as_tensor(req).to(DEV),
                                    positions=None if pos is None else torch.as_tensor(pos).to(DEV))
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


def _check_compaction(got, hid):
    """The compaction part against the oracle's compaction of the fused
    call's own accepted lengths and tokens."""
    acc = got["accepted_len"].numpy()
    ot = got["out_tokens"].numpy()
    bits = hid.contiguous().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.compact(bits, acc, ot, None)
    n = int(ref["offsets"][-1])
    assert got["offsets"].numpy().tolist() == ref["offsets"].tolist()
    assert np.array_equal(got["next_tokens"].numpy()[:n], ref["next_tokens"])
    g = got["out_hidden"][:n].contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(g, ref["out_hidden"])
    assert ref["dev_error"] == 0


def _check_same_as_verify(got, tgt, drf, d, T, top_p, seed, req, pos):
    import speculative_decoding_verification_60_gb300 as svp

    ref = svp.verify_linear(tgt.to(DEV), None if drf is None else drf.to(DEV),
                            torch.as_tensor(d, dtype=torch.int32).to(DEV), T, top_p, seed,
                            request_ids=None if req is None else torch.as_tensor(req).to(DEV),
                            positions=None if pos is None else torch.as_tensor(pos).to(DEV))
    torch.cuda.synchronize()
    for key in ("accepted_len", "out_tokens", "accept_prob", "token_probs", "len_hist", "dev_error"):
        assert torch.equal(got[key], ref[key].cpu()), key


@pytest.mark.parametrize("T,top_p", [(0.7, 0.9), (1.0, 1.0), (0.0, 1.0)])
@pytest.mark.parametrize("B,k,V,H", [(6, 3, 3000, 64), (11, 5, 4099, 1001), (4, 2, 9000, 7168)])
def test_small_cases(B, k, V, H, T, top_p):
    seed = 9
    tgt, drf, d, req, pos, rows = linear_case(B, k, V, "bf16", T, top_p, data_seed=B * 13 + k, seed=seed)
    hid = synth.hidden_states(B, k + 1, H, seed=B + H)
    got = _fused(tgt, drf, d, hid, T, top_p, seed, req, pos)
    _check_same_as_verify(got, tgt, drf, d, T, top_p, seed, req, pos)
    _check_compaction(got, hid)
    ref = oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows)
    res = {key: v.numpy() for key, v in got.items() if v.dtype != torch.bfloat16}
    excused = compare_linear(res, ref, rows, greedy=(T == 0.0), label=f"fused T={T} p={top_p}",
                             margin_of=lambda b, i: row_topp_margin(tgt, drf, b, i, T, top_p))
    assert excused <= 1


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_full_size_workload(T):
    """B=1024, k=3, V=129280 with the 7168-wide hidden states (DeepSeek-scale
    MTP verification), sampled and greedy."""
    w = synth.WORKLOADS["linear-b1024-k3-v129280-h7168"]
    B, k, V, H = w["B"], w["k"], w["V"], w["H"]
    tgt, drf = synth.linear_logits(B, k, V, "bf16", w["data_seed"], device="cuda")
    d = torch.argmax(drf.float(), dim=-1).to(torch.int32) if T == 0 else \
        synth.uniform_tokens((B, k), V, w["data_seed"] + 3).to("cuda")
    hid = synth.hidden_states(B, k + 1, H, seed=w["data_seed"], device="cuda")
    req = np.arange(B, dtype=np.int64) + 100
    pos = np.full(B, 77, dtype=np.int64)
    got = _fused(tgt, drf, d, hid, T, 1.0, w["seed"], req, pos)
    _check_same_as_verify(got, tgt, drf, d.cpu().numpy(), T, 1.0, w["seed"], req, pos)
    _check_compaction(got, hid.cpu())


def test_mtp_shift_golden_through_the_fused_call():
    """The hand-made §MTP shift (tests/golden/compact_mtp_shift.json),
    reached through greedy verification: logits built so that request b
    accepts exactly accepted_len[b] drafts and emits out_tokens[b]."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "compact_mtp_shift.json")))
    B, T, H = g["B"], g["T"], g["H"]
    k, V = T - 1, 64
    tgt = torch.zeros(B, k + 1, V)
    d = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        a = g["accepted_len"][b]
        toks = g["out_tokens"][b]
        for i in range(k + 1):
            x = toks[i] if i <= a else 1  # rows past the emitted token: any argmax
            tgt[b, i, x] = 5.0
        for i in range(k):
            # drafts 1..a equal the argmax of the row before; draft a+1 differs
            d[b, i] = toks[i] if i < a else (toks[i] + 1 if i == a else 2)
    tgt = tgt.to(torch.bfloat16)
    hid = np.zeros((B, T, H), dtype=np.uint16)
    for b in range(B):
        for r in range(T):
            hid[b, r] = [100 * b + 10 * r, 100 * b + 10 * r + 1]
    h = torch.from_numpy(hid.view(np.int16)).view(torch.bfloat16)
    got = _fused(tgt, None, d, h, 0.0, 1.0, 0)
    assert got["accepted_len"].tolist() == g["accepted_len"]
    assert got["offsets"].tolist() == g["expect_offsets"]
    assert got["next_tokens"][:7].tolist() == g["expect_next_tokens"]
    assert got["out_hidden"][:7].view(torch.int16).numpy().view(np.uint16).tolist() == g["expect_rows"]
