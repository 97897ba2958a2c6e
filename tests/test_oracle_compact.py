"""Pins of the oracle's compaction against a hand-made fixture of the
one-step token/hidden-state shift ("Accelerating Sonar through speculation",
§MTP and §MTP schedule for a single token)."""

import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "compact_mtp_shift.json")


def _fixture():
    g = json.load(open(GOLDEN))
    B, T, H = g["B"], g["T"], g["H"]
    hid = np.zeros((B, T, H), dtype=np.uint16)
    for b in range(B):
        for r in range(T):
            hid[b, r] = [100 * b + 10 * r, 100 * b + 10 * r + 1]
    return g, hid


def test_linear_compaction_golden():
    g, hid = _fixture()
    out = oracle.compact(hid, g["accepted_len"], g["out_tokens"])
    assert out["offsets"].tolist() == g["expect_offsets"]
    assert out["next_tokens"].tolist() == g["expect_next_tokens"]
    assert out["out_hidden"].tolist() == g["expect_rows"]
    assert out["dev_error"] == 0


def test_tree_compaction_golden():
    g, hid = _fixture()
    out = oracle.compact(hid, g["accepted_len"], g["out_tokens"], g["tree_path_nodes"])
    assert out["offsets"].tolist() == g["expect_offsets"]
    assert out["out_hidden"].tolist() == g["expect_tree_rows"]


def test_bad_lengths_contribute_nothing():
    g, hid = _fixture()
    out = oracle.compact(hid, [1, 9, -1], g["out_tokens"])
    assert out["offsets"].tolist() == [0, 2, 2, 2]
    assert out["dev_error"] == oracle.ERR_LENGTH
