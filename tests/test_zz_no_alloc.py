"""spec_verify_linear_noalloc, the variant for callers that cannot allocate
device memory where they verify (code inside an allocator or a memory pool,
code whose device memory is fixed at start-up).  It must give the same
results as spec_verify_linear, call after call, while allocating nothing
itself: the test allocates every input and output up front.

This file sorts last so that a run stopping at its first failure has run
every other test before it; it also passes on its own in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_60_gb300 import build

    build.build()
    import speculative_decoding_verification_60_gb300 as svp

    return svp


def _inputs(seed, B=12, k=4, V=5000, T=0.8):
    import synth

    from gpu_parity import draft_tokens_from_oracle

    tgt, drf = synth.linear_logits(B, k, V, "bf16", data_seed=seed)
    if B > 64:  # many requests: uniform drafts (the comparison is with the workspace call)
        d = synth.uniform_tokens((B, k), V, seed).numpy()
    else:
        d = draft_tokens_from_oracle(drf, T if T > 0 else 1.0, 0.9, seed=seed)
    dev = torch.device("cuda:0")
    return (tgt.to(dev), drf.to(dev), torch.from_numpy(d).to(dev),
            torch.arange(B, dtype=torch.int64, device=dev) + 7, torch.full((B,), 40, dtype=torch.int64, device=dev))


def _noalloc(svp, tgt, drf, d, req, pos, T, top_p, seed, out=None):
    B, k1, V = tgt.shape
    k = k1 - 1
    dev = tgt.device
    out = out or dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty(B, k + 1, dtype=torch.int32, device=dev),
               accept_prob=torch.empty(B, k, dtype=torch.float32, device=dev),
               token_probs=torch.empty(B, k, 2, dtype=torch.float32, device=dev),
               len_hist=torch.empty(k + 1, dtype=torch.int32, device=dev),
               dev_error=torch.empty(1, dtype=torch.int32, device=dev))
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    sp = svp.SamplingParams(T, top_p, seed, 0)
    st = svp.load().spec_verify_linear_noalloc(
        P(tgt), P(drf), 0, P(d), B, k, V, P(req), P(pos), ctypes.byref(sp), P(out["accepted_len"]),
        P(out["out_tokens"]), P(out["accept_prob"]), P(out["token_probs"]), P(out["len_hist"]), P(out["dev_error"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, svp.status_string(st)
    return out


@pytest.mark.parametrize("B,k,V", [(12, 4, 5000), (21845, 1, 64)])
def test_noalloc_matches_workspace_call_twice_in_a_row(lib, B, k, V):
    """Sampled with top-p, sampled without it, and greedy, each called twice
    on the same array; (21845, 1, 64) fills 65535 of its 65536 rows (no odd
    row count reaches 65536 itself)."""
    svp = lib
    for seed, (T, top_p) in ((21, (0.8, 0.9)), (22, (1.0, 1.0)), (23, (0.0, 1.0))):
        tgt, drf, d, req, pos = _inputs(seed, B=B, k=k, V=V, T=T)
        got = _noalloc(svp, tgt, drf, d, req, pos, T, top_p, seed)
        ref = svp.verify_linear(tgt, drf, d, T, top_p, seed, request_ids=req, positions=pos)
        torch.cuda.synchronize()
        for key in ("accepted_len", "out_tokens", "len_hist", "dev_error"):
            assert torch.equal(got[key], ref[key]), key
        for key in ("accept_prob", "token_probs"):
            np.testing.assert_allclose(got[key].cpu().numpy(), ref[key].cpu().numpy(), atol=1e-5, rtol=0)


def test_noalloc_rejects_batches_above_its_limit(lib):
    svp = lib
    sp = svp.SamplingParams(1.0, 1.0, 0, 0)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    P = ctypes.c_void_p(x.data_ptr())
    # 4096 * (2*8 + 1) = 69632 rows > 65536: refused before any work is enqueued
    st = svp.load().spec_verify_linear_noalloc(P, P, 0, P, 4096, 8, 8, None, None, ctypes.byref(sp), P, P,
                                               None, None, None, None, None)
    assert svp.status_string(st) == "SPEC_ERR_UNSUPPORTED"


def test_noalloc_allocates_no_device_memory(lib):
    """After a first call on the device (which looks up the array), further
    calls leave the device's free memory as it was."""
    svp = lib
    tgt, drf, d, req, pos = _inputs(31, B=16, k=3, V=3000, T=0.9)
    out = _noalloc(svp, tgt, drf, d, req, pos, 0.9, 0.9, 5)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(svp, tgt, drf, d, req, pos, 0.9, 0.9, 5, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
