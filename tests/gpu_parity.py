"""Shared helpers of the GPU parity tests: seeded cases fed to both the CUDA
path (through the C ABI) and the oracle, and element-by-element checks.

Bar (floating point decides integers here): greedy results bit-exact;
sampled per-token probabilities within 1e-5 absolute; decisions identical
except requests whose oracle decision margin is < 1e-6, which are counted.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

PROB_TOL = 1e-5
MARGIN = 1e-6

# The oracle numbers its error bits its own way; the C ABI's are
# SPEC_DEVERR_TOKEN 1, NONFINITE 2, PARENT 4, LENGTH 8.
_TO_SPEC = {oracle.ERR_TOKEN: 1, oracle.ERR_NONFINITE: 2, oracle.ERR_PARENT: 4, oracle.ERR_LENGTH: 8}


def spec_bits(oracle_bits: int) -> int:
    out = 0
    for ob, sb in _TO_SPEC.items():
        if oracle_bits & ob:
            out |= sb
    return out


def draft_tokens_from_oracle(drf, T, top_p, seed, rows=None):
    """Draft tokens d_{i+1} ~ filter(softmax(draft row i / T)) drawn by the
    oracle (drafts are the draft model's samples; greedy when T == 0)."""
    B, k, V = drf.shape
    d = np.zeros((B, k), dtype=np.int32)
    for b in (range(B) if rows is None else rows):
        row = drf[b].cpu() if isinstance(drf, torch.Tensor) else drf[b]
        d[b] = oracle.sample_rows(row, T, top_p, seed=seed, req=np.full(k, b), pos=np.arange(k))
    return d


def run_gpu_linear(tgt, drf, d, T, top_p, seed, req, pos):
    import speculative_decoding_verification_60_gb300 as svp

    dev = torch.device("cuda:0")
    out = svp.verify_linear(tgt.to(dev), None if drf is None else drf.to(dev),
                            torch.as_tensor(d, dtype=torch.int32).to(dev), T, top_p, seed,
                            request_ids=torch.as_tensor(req, dtype=torch.int64).to(dev),
                            positions=torch.as_tensor(pos, dtype=torch.int64).to(dev))
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def row_topp_margin(tgt, drf, b, i, T, top_p) -> float:
    """Smaller oracle top-p margin of target row i and draft row i of
    request b: how far, in probability mass, the nucleus boundary of those
    rows is from top_p."""
    m = np.inf
    for rows in (tgt, drf):
        if rows is None or T == 0.0:
            continue
        row = rows[b, i].cpu() if isinstance(rows, torch.Tensor) else rows[b, i]
        m = min(m, oracle.row_probs(row, T, top_p)[2])
    return m


def compare_linear(got, ref, rows, greedy: bool, label: str = "", margin_of=None, log=None) -> int:
    """Compare the GPU result for the batch rows `rows` with the oracle run
    on exactly those rows (ref indexed 0..len(rows)-1).  Returns the number
    of margin-excused mismatches.  margin_of(b, i), when given, is the
    top-p margin of drafted position i's rows (a boundary one token apart
    shifts every probability of the row).  log, when given, receives one
    (request, kind, margin) entry per excused mismatch."""
    excused = 0
    for j, b in enumerate(rows):
        ga, ra = int(got["accepted_len"][b]), int(ref["accepted_len"][j])
        gt, rt = got["out_tokens"][b], ref["out_tokens"][j]
        same = ga == ra and np.array_equal(gt, rt)
        if greedy:
            assert same, f"{label} request {b}: gpu a={ga} {gt.tolist()} oracle a={ra} {rt.tolist()}"
        else:
            if not same:
                assert ref["margin"][j] < MARGIN, (
                    f"{label} request {b}: gpu a={ga} {gt.tolist()} oracle a={ra} {rt.tolist()} "
                    f"margin {ref['margin'][j]:.3g}")
                excused += 1
                if log is not None:
                    log.append((b, "decision", float(ref["margin"][j])))
            tp = got["token_probs"][b].astype(np.float64)
            err = np.max(np.abs(tp - ref["tok_p"][j])) if tp.size else 0.0
            if err >= PROB_TOL:
                # a nucleus boundary one token apart moves every probability
                # of the row; allowed only at a rounding-sized margin
                bad_pos = np.nonzero(np.max(np.abs(tp - ref["tok_p"][j]), axis=1) >= PROB_TOL)[0]
                for i in bad_pos:
                    mg = margin_of(b, int(i)) if margin_of is not None else ref["margin"][j]
                    assert mg < MARGIN, f"{label} request {b} pos {i}: token probability error {err:.3g}, margin {mg:.3g}"
                    if log is not None:
                        log.append((b, "token probability", float(mg)))
                excused += int(same)
            # accept_prob = min(1, p/q): consistent with the GPU's own p and q,
            # and close to the oracle's in relative terms (p/q amplifies q's error)
            ap = got["accept_prob"][b].astype(np.float64)
            p_, q_ = tp[:, 0], tp[:, 1]
            own = np.where(q_ > 0, np.minimum(1.0, p_ / np.where(q_ > 0, q_, 1.0)), 0.0)
            assert np.allclose(ap, own, rtol=1e-6, atol=1e-7), f"{label} request {b}: accept_prob != min(1, p/q)"
            aerr = np.abs(ap - ref["accept_prob"][j])
            ok = aerr <= PROB_TOL + 1e-4 * ref["accept_prob"][j]
            for i in np.nonzero(~ok)[0]:
                mg = margin_of(b, int(i)) if margin_of is not None else ref["margin"][j]
                assert mg < MARGIN, f"{label} request {b} pos {i}: accept probability error {aerr.max():.3g}"
        if greedy:
            assert np.array_equal(got["accept_prob"][b], ref["accept_prob"][j].astype(np.float32))
    return excused


def linear_case(B, k, V, dtype, T, top_p, data_seed, seed, device="cpu", check_rows=None, draft_seed=5):
    """Inputs of one linear case: logits per the workload recipe, drafts
    from the oracle's draft sampler for the checked rows (uniform random
    tokens elsewhere), request ids and positions that differ from the slot."""
    tgt, drf = synth.linear_logits(B, k, V, dtype, data_seed, device=device)
    rows = list(range(B)) if check_rows is None else list(check_rows)
    d = synth.uniform_tokens((B, k), V, data_seed + 7).numpy()
    sub = draft_tokens_from_oracle(drf[rows], T, top_p, draft_seed)
    for j, b in enumerate(rows):
        d[b] = sub[j]
    req = np.arange(B, dtype=np.int64) * 3 + 11
    pos = (np.arange(B, dtype=np.int64) * 7) % 1000 + 5
    return tgt, drf, d, req, pos, rows


def oracle_linear(tgt, drf, d, T, top_p, seed, req, pos, rows, chunk: int = 16):
    """The oracle on the batch rows `rows` (processed a few requests at a
    time to bound host memory); results are indexed 0..len(rows)-1."""
    sel = list(rows)
    parts = []
    for c0 in range(0, len(sel), chunk):
        cs = sel[c0:c0 + chunk]
        t = tgt[cs].cpu() if isinstance(tgt, torch.Tensor) else tgt[cs]
        q = None
        if drf is not None and T != 0.0:
            q = drf[cs].cpu() if isinstance(drf, torch.Tensor) else drf[cs]
        parts.append(oracle.verify_linear(t, q, d[cs], T, top_p, seed, req_ids=req[cs], positions=pos[cs]))
    out = {}
    for key in parts[0]:
        if key == "len_hist":
            out[key] = sum(p[key] for p in parts)
        elif key == "dev_error":
            err = 0
            for p in parts:
                err |= p[key]
            out[key] = err
        else:
            out[key] = np.concatenate([p[key] for p in parts])
    return out
