"""Pins of the oracle's tree verification ("Accelerating Sonar through
speculation", §EAGLE: Top-K candidates per node, the longest accepted path
plus one target token; children tested in turn with residual updates)."""

import numpy as np
import pytest

import oracle
import synth
from exact_enum import ToyWorld, max_abs_diff, tree_emitted_distribution

TREES = {
    "full-k2-d2": [-1, 0, 0, 1, 1, 2, 2],
    "pruned": [-1, 0, 0, 1],
    "k3-d1": [-1, 0, 0, 0],
    "chain": [-1, 0, 1],
}


@pytest.mark.parametrize("mode", [oracle.CHILD_WOR, oracle.CHILD_IID, oracle.CHILD_DET])
@pytest.mark.parametrize("tree", sorted(TREES))
def test_tree_emitted_distribution_equals_target_exactly(mode, tree):
    parent = TREES[tree]
    V = 4 if tree == "k3-d1" else 3
    w = ToyWorld(V, 2, seed=31 + mode, T=1.0, top_p=1.0)
    dmax, _ = oracle.tree_depths(np.array(parent))
    assert max_abs_diff(tree_emitted_distribution(w, parent, mode), w.target_joint(dmax + 1)) < 1e-12


@pytest.mark.parametrize("mode", [oracle.CHILD_IID, oracle.CHILD_DET])
def test_tree_exact_with_top_p_and_temperature(mode):
    w = ToyWorld(4, 2, seed=5, T=0.8, top_p=0.85)
    parent = TREES["full-k2-d2"]
    assert max_abs_diff(tree_emitted_distribution(w, parent, mode), w.target_joint(3)) < 1e-12


@pytest.mark.parametrize("mode", [oracle.CHILD_WOR, oracle.CHILD_IID])
def test_chain_tree_equals_linear(mode):
    """A tree with one child per node is a linear draft: same outputs for
    the same uniforms (positions follow depth)."""
    rng = np.random.default_rng(40 + mode)
    B, k, V = 40, 3, 7
    tgt = rng.normal(0, 1, (B, k + 1, V))
    drf = rng.normal(0, 1, (B, k + 1, V))
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    tok = np.concatenate([np.zeros((B, 1), np.int32), d], 1)
    parent = np.arange(-1, k, dtype=np.int32)
    for T, tp in ((1.0, 1.0), (0.7, 0.8), (0.0, 1.0)):
        lin = oracle.verify_linear(tgt, drf[:, :k], d, T, tp, seed=17, positions=np.arange(B) * 3)
        tr = oracle.verify_tree(tgt, drf, tok, parent, T, tp, seed=17, mode=mode, positions=np.arange(B) * 3)
        assert np.array_equal(lin["accepted_len"], tr["accepted_len"])
        assert np.array_equal(lin["out_tokens"], tr["out_tokens"])


def test_deterministic_chain_equals_linear_with_one_hot_draft():
    rng = np.random.default_rng(50)
    B, k, V = 30, 3, 6
    tgt = rng.normal(0, 1, (B, k + 1, V))
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    oh = np.full((B, k, V), -np.inf)
    for b in range(B):
        for i in range(k):
            oh[b, i, d[b, i]] = 0.0
    tok = np.concatenate([np.zeros((B, 1), np.int32), d], 1)
    parent = np.arange(-1, k, dtype=np.int32)
    lin = oracle.verify_linear(tgt, oh, d, 1.0, 1.0, seed=8)
    tr = oracle.verify_tree(tgt, None, tok, parent, 1.0, 1.0, seed=8, mode=oracle.CHILD_DET)
    assert np.array_equal(lin["accepted_len"], tr["accepted_len"])
    assert np.array_equal(lin["out_tokens"], tr["out_tokens"])


def test_tree_outputs_are_a_valid_path():
    parent = synth.pruned_tree(4, 5, 60)
    dmax, depth = oracle.tree_depths(parent)
    assert dmax == 5
    rng = np.random.default_rng(60)
    B, N, V = 6, len(parent), 11
    tgt = rng.normal(0, 1, (B, N, V))
    drf = tgt + rng.normal(0, 0.7, (B, N, V))
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    for T in (1.0, 0.0):
        out = oracle.verify_tree(tgt, drf, tok, parent, T, 1.0, seed=1, mode=oracle.CHILD_IID)
        for b in range(B):
            a = out["accepted_len"][b]
            path = out["path_nodes"][b]
            assert path[0] == 0 and np.all(path[a + 1:] == -1)
            for j in range(1, a + 1):
                assert parent[path[j]] == path[j - 1]
                assert out["out_tokens"][b, j - 1] == tok[b, path[j]]
            assert 0 <= out["out_tokens"][b, a] < V


def test_bad_parent_array_is_flagged():
    out = oracle.verify_tree(np.zeros((1, 3, 4)), np.zeros((1, 3, 4)), np.zeros((1, 3), np.int32),
                             np.array([-1, 2, 0], np.int32), 1.0, 1.0, seed=0)
    assert out["dev_error"] & oracle.ERR_PARENT


@pytest.mark.parametrize("mode", [oracle.CHILD_WOR, oracle.CHILD_IID, oracle.CHILD_DET])
def test_a_request_depends_only_on_its_own_tree(mode):
    """Per-request trees (§EAGLE: fixed or dynamically shaped trees) are read
    as the fixed-tree walk applied to each request's own tree.  That reading
    needs a request's result to depend only on its rows, tree, request id
    and position: the batched oracle's result for a request equals the
    oracle on that request alone, and a request keeps its result when the
    other requests of the batch change."""
    rng = np.random.default_rng(60 + mode)
    B, V = 6, 9
    for name, parent in TREES.items():
        N = len(parent)
        tgt = rng.normal(0, 1.2, (B, N, V))
        drf = tgt + rng.normal(0, 0.6, (B, N, V))
        tok = rng.integers(0, V, (B, N)).astype(np.int32)
        req = np.arange(B, dtype=np.int64) * 5 + 2
        pos = np.arange(B, dtype=np.int64) + 7
        for T, tp in ((1.0, 1.0), (0.8, 0.9)):
            batch = oracle.verify_tree(tgt, drf, tok, parent, T, tp, seed=23, mode=mode, req_ids=req, positions=pos)
            other = tgt.copy()
            other[1:] = rng.normal(0, 1.2, other[1:].shape)  # the rest of the batch changes
            batch2 = oracle.verify_tree(other, drf, tok, parent, T, tp, seed=23, mode=mode, req_ids=req,
                                        positions=pos)
            for b in range(B):
                one = oracle.verify_tree(tgt[b:b + 1], drf[b:b + 1], tok[b:b + 1], parent, T, tp, seed=23, mode=mode,
                                         req_ids=req[b:b + 1], positions=pos[b:b + 1])
                for key in ("accepted_len", "path_nodes", "out_tokens"):
                    assert np.array_equal(batch[key][b], one[key][0]), (name, b, key)
                    if b == 0:
                        assert np.array_equal(batch2[key][0], one[key][0]), (name, key)
