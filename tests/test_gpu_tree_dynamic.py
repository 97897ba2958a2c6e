"""GPU parity of spec_verify_tree_dynamic: a tree of its own for every
request ("Accelerating Sonar through speculation", §EAGLE: the tree is
fixed, or dynamically shaped as in the cited EAGLE-2).  Every request must
give what the oracle's tree verification gives for that request alone, with
its own parent array and node count; rows, tokens and parent entries past a
request's nodes hold values that would be errors if they were read."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_parity import MARGIN, spec_bits

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def random_tree(n, max_depth, rng):
    """A parent array of n nodes (parent[i] < i) no deeper than max_depth."""
    parent, depth = [-1], [0]
    for i in range(1, n):
        while True:
            p = int(rng.integers(0, i))
            if depth[p] < max_depth:
                break
        parent.append(p)
        depth.append(depth[p] + 1)
    return parent


def dyn_case(B, Nmax, V, T, top_p, mode, seed, max_depth=4):
    rng = np.random.default_rng(seed)
    counts = rng.integers(1, Nmax + 1, size=B).astype(np.int32)
    counts[0], counts[-1] = 1, Nmax  # a lone root, and a tree of the full size
    parents = np.full((B, Nmax), 12345, dtype=np.int32)  # past a tree's nodes: never read
    for b in range(B):
        parents[b, :counts[b]] = random_tree(int(counts[b]), max_depth, rng)
    tgt, drf = synth.tree_logits(B, Nmax, V, seed)
    tok = synth.uniform_tokens((B, Nmax), V, seed + 2).numpy()
    for b in range(B):
        nb = int(counts[b])
        par = parents[b, :nb]
        for n in range(nb):
            kids = [i for i in range(nb) if par[i] == n]
            if kids:
                draw = oracle.draw_children(drf[b, n].cpu(), T if T > 0 else 1.0, top_p, len(kids), mode,
                                            seed=17, req=b, pos=n)
                for c, x in zip(kids, draw):
                    tok[b, c] = x if x >= 0 else (b * 31 + c * 7) % V
        tok[b, nb:] = -5                 # an invalid token, if it were read
        tgt[b, nb:] = float("nan")       # a non-finite row, if it were read
        drf[b, nb:] = float("nan")
    req = np.arange(B, dtype=np.int64) * 3 + 500
    pos = np.arange(B, dtype=np.int64) * 11 + 2
    return tgt, drf, tok, parents, counts, req, pos


def run_dynamic(tgt, drf, tok, parents, counts, max_depth, T, top_p, seed, mode, req, pos):
    import speculative_decoding_verification_60_gb300 as svp

    out = svp.verify_tree_dynamic(tgt.to(DEV), drf.to(DEV), torch.as_tensor(tok, dtype=torch.int32).to(DEV),
                                  torch.as_tensor(parents).to(DEV), torch.as_tensor(counts).to(DEV), max_depth, T,
                                  top_p, seed, mode, request_ids=torch.as_tensor(req).to(DEV),
                                  positions=torch.as_tensor(pos).to(DEV))
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


@pytest.mark.parametrize("mode", [oracle.CHILD_WOR, oracle.CHILD_IID, oracle.CHILD_DET])
@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 0.9), (0.0, 1.0)])
def test_per_request_trees_match_the_oracle(mode, T, top_p):
    B, Nmax, V, seed, max_depth = 10, 20, 2003, 5, 4
    tgt, drf, tok, parents, counts, req, pos = dyn_case(B, Nmax, V, T, top_p, mode, seed=40 + mode, max_depth=max_depth)
    got = run_dynamic(tgt, drf, tok, parents, counts, max_depth, T, top_p, seed, mode, req, pos)
    assert int(got["dev_error"][0]) == 0
    excused = 0
    for b in range(B):
        nb = int(counts[b])
        ref = oracle.verify_tree(tgt[b:b + 1, :nb].cpu(), drf[b:b + 1, :nb].cpu(), tok[b:b + 1, :nb],
                                 parents[b, :nb], T, top_p, seed, mode=mode, req_ids=req[b:b + 1],
                                 positions=pos[b:b + 1])
        wb = ref["path_nodes"].shape[1]
        same = (got["accepted_len"][b] == ref["accepted_len"][0]
                and np.array_equal(got["path_nodes"][b, :wb], ref["path_nodes"][0])
                and np.array_equal(got["out_tokens"][b, :wb], ref["out_tokens"][0]))
        if not same:
            assert T > 0 and ref["margin"][0] < MARGIN, (
                f"request {b} ({nb} nodes): gpu {got['path_nodes'][b].tolist()} {got['out_tokens'][b].tolist()} "
                f"oracle {ref['path_nodes'][0].tolist()} {ref['out_tokens'][0].tolist()}")
            excused += 1
        # columns past this request's depth stay empty
        assert (got["path_nodes"][b, wb:] == -1).all() and (got["out_tokens"][b, wb:] == -1).all()
    assert excused <= 1


def test_one_request_shape_equals_the_static_call():
    """Every request with the same tree: the per-request call gives the static call's results."""
    import speculative_decoding_verification_60_gb300 as svp

    B, V, T, top_p, seed, mode = 6, 1500, 0.8, 0.95, 3, oracle.CHILD_WOR
    parent = np.array([-1, 0, 0, 1, 1, 2, 3, 3], dtype=np.int32)
    N = len(parent)
    tgt, drf = synth.tree_logits(B, N, V, 77)
    tok = synth.uniform_tokens((B, N), V, 79).to(torch.int32)
    req = torch.arange(B, dtype=torch.int64) + 9
    pos = torch.arange(B, dtype=torch.int64) * 2
    args = dict(request_ids=req.to(DEV), positions=pos.to(DEV))
    st = svp.verify_tree(tgt.to(DEV), drf.to(DEV), tok.to(DEV), torch.as_tensor(parent).to(DEV), 3, T, top_p, seed,
                         mode, **args)
    dy = svp.verify_tree_dynamic(tgt.to(DEV), drf.to(DEV), tok.to(DEV),
                                 torch.as_tensor(np.tile(parent, (B, 1))).to(DEV),
                                 torch.full((B,), N, dtype=torch.int32).to(DEV), 3, T, top_p, seed, mode, **args)
    torch.cuda.synchronize()
    for key in ("accepted_len", "path_nodes", "out_tokens", "dev_error"):
        assert torch.equal(st[key].cpu(), dy[key].cpu()), key


def test_bad_shapes_flag_only_their_request():
    """A node count outside 1..N, or a parent entry not below its node,
    marks that request invalid (defined fallback: a = 0, the argmax of target
    row 0) and leaves the others as they are."""
    B, Nmax, V, T, top_p, seed, mode = 5, 12, 900, 1.0, 1.0, 8, oracle.CHILD_WOR
    tgt, drf, tok, parents, counts, req, pos = dyn_case(B, Nmax, V, T, top_p, mode, seed=71, max_depth=3)
    good = run_dynamic(tgt, drf, tok, parents, counts, 3, T, top_p, seed, mode, req, pos)
    counts2, parents2 = counts.copy(), parents.copy()
    counts2[1] = 0              # no nodes at all
    counts2[2] = Nmax + 1       # more nodes than the inputs hold
    if counts2[3] < 3:
        counts2[3] = 3
        parents2[3, :3] = [-1, 0, 0]
    parents2[3, 2] = 2          # a node that is its own parent
    bad = run_dynamic(tgt, drf, tok, parents2, counts2, 3, T, top_p, seed, mode, req, pos)
    assert int(bad["dev_error"][0]) == spec_bits(oracle.ERR_PARENT)
    for b in (1, 2, 3):
        assert bad["accepted_len"][b] == 0
        assert bad["path_nodes"][b].tolist() == [0, -1, -1, -1]
        assert bad["out_tokens"][b, 0] == oracle.argmax(tgt[b, 0])
    for b in (0, 4):
        for key in ("accepted_len", "path_nodes", "out_tokens"):
            assert np.array_equal(bad[key][b], good[key][b]), (key, b)
