"""GPU parity of spec_verify_tree against the oracle, through the C ABI
("Accelerating Sonar through speculation", §EAGLE)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_parity import MARGIN, spec_bits

pytestmark = pytest.mark.gpu


def tree_case(B, parent, V, dtype, T, top_p, mode, data_seed, rows=None):
    parent = np.asarray(parent, dtype=np.int32)
    N = len(parent)
    if dtype == "f32":
        tgt = synth.gaussian((B, N, V), 2.0, data_seed)
        drf = tgt + synth.gaussian((B, N, V), 0.7, data_seed + 1)
    else:
        tgt, drf = synth.tree_logits(B, N, V, data_seed)
    tok = synth.uniform_tokens((B, N), V, data_seed + 2).numpy()
    children = [[i for i in range(N) if parent[i] == n] for n in range(N)]
    for b in (range(B) if rows is None else rows):
        for n in range(N):
            if children[n]:
                draw = oracle.draw_children(drf[b, n].cpu(), T if T > 0 else 1.0, top_p, len(children[n]), mode,
                                            seed=17, req=b, pos=n)
                for c, x in zip(children[n], draw):
                    # a draw past an exhausted nucleus (WOR) has no token: give
                    # the child one the draft cannot produce (q = 0, rejected)
                    tok[b, c] = x if x >= 0 else (b * 31 + c * 7) % V
    req = np.arange(B, dtype=np.int64) + 1000
    pos = np.arange(B, dtype=np.int64) * 5
    return tgt, drf, tok, parent, req, pos


def run_gpu_tree(tgt, drf, tok, parent, T, top_p, seed, mode, req, pos, max_depth=None):
    import speculative_decoding_verification_60_gb300 as svp

    dev = torch.device("cuda:0")
    dmax = oracle.tree_depths(parent)[0] if max_depth is None else max_depth
    out = svp.verify_tree(tgt.to(dev), drf.to(dev), torch.as_tensor(tok, dtype=torch.int32).to(dev),
                          torch.as_tensor(parent, dtype=torch.int32).to(dev), dmax, T, top_p, seed, mode,
                          request_ids=torch.as_tensor(req).to(dev), positions=torch.as_tensor(pos).to(dev))
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def compare_tree(tgt, drf, tok, parent, T, top_p, seed, mode, req, pos, rows, label):
    got = run_gpu_tree(tgt, drf, tok, parent, T, top_p, seed, mode, req, pos)
    excused = 0
    for b in rows:
        ref = oracle.verify_tree(tgt[b:b + 1].cpu(), drf[b:b + 1].cpu(), tok[b:b + 1], parent, T, top_p, seed,
                                 mode=mode, req_ids=req[b:b + 1], positions=pos[b:b + 1])
        same = (got["accepted_len"][b] == ref["accepted_len"][0]
                and np.array_equal(got["path_nodes"][b], ref["path_nodes"][0])
                and np.array_equal(got["out_tokens"][b], ref["out_tokens"][0]))
        if not same:
            assert T > 0 and ref["margin"][0] < MARGIN, (
                f"{label} request {b}: gpu {got['path_nodes'][b].tolist()} {got['out_tokens'][b].tolist()} "
                f"oracle {ref['path_nodes'][0].tolist()} {ref['out_tokens'][0].tolist()} margin {ref['margin'][0]:.3g}")
            excused += 1
    return got, excused


TREES = {
    "k2-d2": [-1, 0, 0, 1, 1, 2, 2],
    "pruned": [-1, 0, 0, 1, 3, 3, 2],
    "chain": [-1, 0, 1, 2],
    "wide": [-1] + [0] * 6,
}


@pytest.mark.parametrize("mode", [oracle.CHILD_WOR, oracle.CHILD_IID, oracle.CHILD_DET])
@pytest.mark.parametrize("tree", sorted(TREES))
@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 0.9), (0.0, 1.0)])
def test_small_trees_match_oracle(mode, tree, T, top_p):
    B, V = 12, 777
    args = tree_case(B, TREES[tree], V, "bf16", T, top_p, mode, data_seed=300 + len(TREES[tree]))
    got, excused = compare_tree(*args[:4], T, top_p, 5, mode, args[4], args[5], range(B), f"{tree}/{mode}")
    assert excused <= 1
    assert int(got["dev_error"][0]) == 0


def test_fp32_tree():
    B, V = 6, 3001
    args = tree_case(B, TREES["k2-d2"], V, "f32", 0.9, 0.9, oracle.CHILD_WOR, data_seed=5)
    compare_tree(*args[:4], 0.9, 0.9, 5, oracle.CHILD_WOR, args[4], args[5], range(B), "f32")


@pytest.mark.parametrize("T,top_p,mode", [(1.0, 1.0, oracle.CHILD_WOR), (0.0, 1.0, oracle.CHILD_WOR),
                                          (0.7, 0.9, oracle.CHILD_IID)])
def test_full_size_tree_workload(T, top_p, mode):
    w = synth.WORKLOADS["tree-b32-n60-k4-d5-v128256"]
    parent = synth.pruned_tree(w["K"], w["depth"], w["N"])
    rows = [0, 13, 31]
    args = tree_case(w["B"], parent, w["V"], "bf16", T, top_p, mode, w["data_seed"], rows=rows)
    got, excused = compare_tree(*args[:4], T, top_p, w["seed"], mode, args[4], args[5], rows, "tree-full")
    assert excused <= 1
    assert np.all(got["accepted_len"] <= 5)


def test_bad_parent_and_tokens_are_flagged():
    B, V = 3, 300
    parent = np.array([-1, 0, 0, 1], dtype=np.int32)
    tgt, drf, tok, parent, req, pos = tree_case(B, parent, V, "bf16", 1.0, 1.0, oracle.CHILD_IID, data_seed=9)
    tok[1, 3] = V + 1
    got = run_gpu_tree(tgt, drf, tok, parent, 1.0, 1.0, 5, oracle.CHILD_IID, req, pos)
    assert int(got["dev_error"][0]) & spec_bits(oracle.ERR_TOKEN)
    assert got["accepted_len"][1] == 0 and got["out_tokens"][1, 0] == oracle.argmax(tgt[1, 0])
    bad_parent = np.array([-1, 0, 3, 1], dtype=np.int32)
    got = run_gpu_tree(tgt, drf, tok, bad_parent, 1.0, 1.0, 5, oracle.CHILD_IID, req, pos, max_depth=2)
    assert int(got["dev_error"][0]) & spec_bits(oracle.ERR_PARENT)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_more_children_than_tested_is_flagged_in_every_mode(T):
    """A node with 65 children (the kernel tests at most 64 per node) is
    reported as a bad tree in greedy and sampled mode alike, and the request
    takes the defined fallback (nothing accepted, the argmax of row 0)."""
    B, V, N = 2, 128, 66
    parent = np.array([-1] + [0] * (N - 1), dtype=np.int32)
    tgt, drf = synth.tree_logits(B, N, V, 23)
    tok = np.zeros((B, N), dtype=np.int32)
    tok[:, 1:] = np.arange(N - 1) % V
    tok[:, N - 1] = oracle.argmax(tgt[0, 0])  # greedy would accept the 65th child
    req = np.arange(B, dtype=np.int64)
    pos = np.zeros(B, dtype=np.int64)
    got = run_gpu_tree(tgt, drf, tok, parent, T, 1.0, 7, oracle.CHILD_IID, req, pos)
    assert int(got["dev_error"][0]) & spec_bits(oracle.ERR_PARENT)
    for b in range(B):
        assert got["accepted_len"][b] == 0
        assert got["out_tokens"][b, 0] == oracle.argmax(tgt[b, 0])
