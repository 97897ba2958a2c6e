"""Brute-force enumeration of the exact output distribution of the oracle's
verification, for tiny vocabularies.

The oracle's single-request cores take their uniforms as explicit inputs and
report, in a trace, the threshold each accept test compared against and the
weights of the final draw.  Steering the uniforms (0 forces an accept when
the threshold is positive; the largest double below 1 forces a reject when
it is below 1) walks every decision path of the oracle's own composition.
Each path's probability is the product of min(1, r) or 1 - min(1, r) over
its tests, times the final draw's normalised weight; the draw itself is
pinned separately as an exact inverse CDF.

The reference for the emitted tokens is the target distribution computed
here independently (scipy softmax and the tie-aware top-p definition); the
claim checked is the cited work's: the emitted tokens are distributed
exactly as samples from the target ("Accelerating Sonar through
speculation", §Speculative decoding, §Target-Draft, §EAGLE).
"""

from __future__ import annotations

import itertools

import numpy as np
from scipy.special import softmax

import oracle

U_REJECT = float(np.nextafter(1.0, 0.0))


def ref_probs(x, T: float, top_p: float) -> np.ndarray:
    """Filtered softmax from the definitions, independent of the oracle:
    token v is kept iff the mass of the tokens ranked before it (higher
    logit, or equal logit and lower index) is < top_p."""
    x = np.asarray(x, dtype=np.float64)
    p = softmax(x / T)
    if top_p >= 1.0:
        return p
    V = len(x)
    keep = np.zeros(V, dtype=bool)
    for v in range(V):
        before = sum(p[w] for w in range(V) if x[w] > x[v] or (x[w] == x[v] and w < v))
        keep[v] = before < top_p
    q = np.where(keep, p, 0.0)
    return q / q.sum()


class ToyWorld:
    """Prefix-dependent toy target and draft models over a tiny vocabulary:
    one logit row per prefix, for every prefix up to a given length."""

    def __init__(self, V: int, depth: int, seed: int, T: float, top_p: float, q_equals_p: bool = False,
                 integer_logits: bool = False):
        rng = np.random.default_rng(seed)
        self.V, self.T, self.top_p = V, T, top_p
        self.P, self.Q = {}, {}
        for L in range(depth + 1):
            for pre in itertools.product(range(V), repeat=L):
                if integer_logits:
                    xp = rng.integers(-2, 3, V).astype(np.float64)
                    xq = rng.integers(-2, 3, V).astype(np.float64)
                else:
                    xp = rng.normal(0.0, 1.5, V)
                    xq = xp + rng.normal(0.0, 0.8, V)
                self.P[pre] = xp
                self.Q[pre] = xp.copy() if q_equals_p else xq

    def p(self, pre):
        return ref_probs(self.P[tuple(pre)], self.T, self.top_p)

    def q(self, pre):
        return ref_probs(self.Q[tuple(pre)], self.T, self.top_p)

    def target_joint(self, n: int) -> dict:
        """Exact target probability of every token sequence of length n."""
        out = {}
        for seq in itertools.product(range(self.V), repeat=n):
            pr = 1.0
            for j in range(n):
                pr *= self.p(seq[:j])[seq[j]]
            out[seq] = pr
        return out

    def complete(self, block, n: int, weight: float, acc: dict):
        """Add `weight` times the target probability of every completion of
        `block` to length n into acc."""
        block = tuple(int(t) for t in block)
        rest = n - len(block)
        for tail in itertools.product(range(self.V), repeat=rest):
            seq = block + tail
            pr = weight
            for j in range(len(block), n):
                pr *= self.p(seq[:j])[seq[j]]
            acc[seq] = acc.get(seq, 0.0) + pr


class ThresholdMismatch(AssertionError):
    """The oracle's accept test did not behave as u < threshold."""


def _paths(run_with):
    """Depth-first walk of every decision path.  run_with(us) runs the
    oracle with the uniforms of its first len(us) accept tests set to us and
    the rest steered to accept; it returns the result with a 'trace'.

    Every decision met is also probed just below and just above its traced
    threshold r (when 0 < r < 1), so the comparison itself, not only the
    threshold, is checked to be u < r."""
    stack = [[]]
    probed = set()
    while stack:
        forced = stack.pop()
        us = [0.0 if f else U_REJECT for f in forced]
        out = run_with(us)
        tr = out["trace"]
        dec = tr["accepted"]
        if len(dec) < len(forced) or any(bool(dec[i]) != forced[i] for i in range(len(forced))):
            continue
        for i, r in enumerate(tr["ratio"]):
            key = tuple(bool(x) for x in dec[:i])
            if key in probed or not (0.0 < r < 1.0):
                continue
            probed.add(key)
            prefix = [0.0 if x else U_REJECT for x in dec[:i]]
            lo = run_with(prefix + [r * (1.0 - 1e-9)])["trace"]["accepted"]
            hi = run_with(prefix + [min(r * (1.0 + 1e-9), U_REJECT)])["trace"]["accepted"]
            if not (len(lo) > i and lo[i]) or not (len(hi) > i and not hi[i]):
                raise ThresholdMismatch(f"decision {i}: threshold {r}")
        w = 1.0
        for r, a in zip(tr["ratio"], dec):
            pa = min(1.0, r)
            w *= pa if a else (1.0 - pa)
        if w > 0.0:
            yield w, out
        for i in range(len(forced), len(dec)):
            if dec[i]:
                stack.append([bool(x) for x in dec[:i]] + [False])


def final_dist(out) -> np.ndarray:
    w = np.asarray(out["trace"]["final_w"], dtype=np.float64)
    return w / w.sum()


def linear_emitted_distribution(world: ToyWorld, k: int) -> dict:
    """Exact distribution of the oracle's linear verification output,
    completed with target samples to length k+1, with drafts drawn from the
    (filtered) draft model."""
    V, T, top_p = world.V, world.T, world.top_p
    acc = {}
    for d in itertools.product(range(V), repeat=k):
        pd = 1.0
        for i in range(k):
            pd *= world.q(d[:i])[d[i]]
        if pd == 0.0:
            continue
        tgt = np.stack([world.P[d[:i]] for i in range(k + 1)])
        drf = np.stack([world.Q[d[:i]] for i in range(k)])

        def run_with(us, tgt=tgt, drf=drf, d=d):
            u = [0.0] * k
            for i, x in enumerate(us):
                u[i] = x
            return oracle.linear_request(tgt, drf, np.array(d), T, top_p, u, [0.5] * k, 0.5, want_trace=True)

        for w, out in _paths(run_with):
            a = out["a"]
            fd = final_dist(out)
            for t in range(V):
                if fd[t] > 0.0:
                    world.complete(tuple(d[:a]) + (t,), k + 1, pd * w * fd[t], acc)
    return acc


def _child_assignments(world: ToyWorld, parent, mode: int, K: int):
    """Every assignment of tokens to non-root nodes with its probability
    under the child-drawing mode (WOR, IID, or deterministic top-K)."""
    N = len(parent)
    children = [[i for i in range(N) if parent[i] == n] for n in range(N)]
    prefix = {0: ()}
    order = list(range(N))

    def rec(idx_node, tok, prob):
        if idx_node == N:
            yield list(tok), prob
            return
        n = order[idx_node]
        ch = children[n]
        if not ch:
            yield from rec(idx_node + 1, tok, prob)
            return
        pre = prefix[n]
        q = world.q(pre)
        if mode == oracle.CHILD_DET:
            xq = world.Q[pre]
            ranked = sorted(range(world.V), key=lambda v: (-xq[v], v))
            for j, c in enumerate(ch):
                tok[c] = ranked[j]
                prefix[c] = pre + (ranked[j],)
            yield from rec(idx_node + 1, tok, prob)
            return
        for combo in itertools.product(range(world.V), repeat=len(ch)):
            pr = 1.0
            if mode == oracle.CHILD_IID:
                for x in combo:
                    pr *= q[x]
            else:
                used = 0.0
                seen = set()
                for x in combo:
                    if x in seen or 1.0 - used <= 0.0:
                        pr = 0.0
                        break
                    pr *= q[x] / (1.0 - used)
                    used += q[x]
                    seen.add(x)
            if pr == 0.0:
                continue
            for c, x in zip(ch, combo):
                tok[c] = x
                prefix[c] = pre + (x,)
            yield from rec(idx_node + 1, tok, prob * pr)

    yield from rec(0, [0] * N, 1.0)


def tree_emitted_distribution(world: ToyWorld, parent, mode: int) -> dict:
    """Exact distribution of the oracle's tree verification output,
    completed with target samples to length Dmax+1, with children drawn per
    mode from the draft model at their parent."""
    parent = np.asarray(parent, dtype=np.int32)
    N = len(parent)
    dmax, depth = oracle.tree_depths(parent)
    K = max(int(np.sum(parent == n)) for n in range(N))
    V, T, top_p = world.V, world.T, world.top_p
    acc = {}
    for tok, ptok in _child_assignments(world, parent, mode, K):
        prefix = [()] * N
        for i in range(1, N):
            prefix[i] = prefix[parent[i]] + (tok[i],)
        tgt = np.stack([world.P[prefix[n]] for n in range(N)])
        drf = np.stack([world.Q[prefix[n]] for n in range(N)])

        def run_with(us, tgt=tgt, drf=drf, tok=tok):
            # decisions walk (depth, child round): an accept descends, a
            # reject moves to the next child; the decided outcome of a probed
            # (last) entry does not matter for the placement of later ones
            u_acc = np.zeros((dmax + 1, K))
            dd, j = 0, 0
            for x in us:
                u_acc[dd, j] = x
                if x == 0.0:
                    dd, j = dd + 1, 0
                else:
                    j += 1
            return oracle.tree_request(tgt, drf, np.array(tok), parent, T, top_p, mode, u_acc,
                                       np.full(dmax + 1, 0.5), np.full(dmax + 1, 0.5), want_trace=True)

        for w, out in _paths(run_with):
            a = out["a"]
            fd = final_dist(out)
            path_tokens = tuple(int(x) for x in out["tokens"][:a])
            for t in range(V):
                if fd[t] > 0.0:
                    world.complete(path_tokens + (t,), dmax + 1, ptok * w * fd[t], acc)
    return acc


def max_abs_diff(dist: dict, ref: dict) -> float:
    keys = set(dist) | set(ref)
    return max(abs(dist.get(s, 0.0) - ref.get(s, 0.0)) for s in keys)
