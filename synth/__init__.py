"""Seeded synthetic inputs shaped like the workloads of "Accelerating Sonar
through speculation" (Llama-1B draft / 70B-class target, DeepSeek-scale).

This module only draws random numbers and arranges them into tensors.  It
holds none of the verification method's arithmetic (no softmax, no
filtering, no acceptance rule, no sampling from model distributions); both
the CUDA path and the oracle consume what it returns.

Recipe (each a reading of a workload description):
  * "Zipf" logits: N(0, 1) plus a bias of 8 * r^-1.1, where r in 1..V is the
    token's rank in an independent random permutation of the vocabulary per
    row (rank 1 gets +8).  Rounded to bf16 once.
  * draft logits: bf16(fp32(target_bf16) + N(0, sigma)), sigma = 0.7.
  * tiny fp32 case: target N(0, sigma=2), draft = target + N(0, 0.5).
  * tree: full top-K (K=4) tree of depth 5 pruned to the best N=60 nodes by
    score prod(1/(rank+1)) along the path, ties by BFS order, numbered in BFS
    order so that parent[i] < i.
  * hidden states: N(0, 1) in bf16.
"""

from __future__ import annotations

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zipf_logits(rows: int, V: int, seed: int, device="cpu", chunk: int = 512) -> torch.Tensor:
    """[rows, V] bf16: N(0,1) + 8 * rank^-1.1 with a per-row random rank."""
    device = torch.device(device)
    g = _gen(seed, device)
    out = torch.empty(rows, V, dtype=torch.bfloat16, device=device)
    ranked_bias = 8.0 * torch.arange(1, V + 1, device=device, dtype=torch.float32).pow(-1.1)
    for r0 in range(0, rows, chunk):
        n = min(chunk, rows - r0)
        base = torch.randn(n, V, generator=g, device=device, dtype=torch.float32)
        perm = torch.rand(n, V, generator=g, device=device).argsort(dim=1)
        bias = torch.empty(n, V, device=device, dtype=torch.float32)
        bias.scatter_(1, perm, ranked_bias.expand(n, V))
        out[r0:r0 + n] = (base + bias).to(torch.bfloat16)
    return out


def add_noise(x: torch.Tensor, sigma: float, seed: int, chunk: int = 512) -> torch.Tensor:
    """x + N(0, sigma) computed in fp32 and rounded back to x's dtype."""
    g = _gen(seed, x.device)
    flat = x.reshape(-1, x.shape[-1])
    out = torch.empty_like(flat)
    for r0 in range(0, flat.shape[0], chunk):
        n = min(chunk, flat.shape[0] - r0)
        noise = torch.randn(n, flat.shape[1], generator=g, device=x.device, dtype=torch.float32) * sigma
        out[r0:r0 + n] = (flat[r0:r0 + n].float() + noise).to(x.dtype)
    return out.reshape(x.shape)


def gaussian(shape, sigma: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    g = _gen(seed, torch.device(device))
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * sigma).to(dtype)


def uniform_tokens(shape, V: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, torch.device(device))
    return torch.randint(0, V, tuple(shape), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def hidden_states(B: int, T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    return gaussian((B, T, H), 1.0, seed, device, torch.bfloat16)


def pruned_tree(K: int = 4, depth: int = 5, N: int = 60) -> np.ndarray:
    """Parent array (int32, BFS order, parent[0] = -1) of the N best nodes
    of a full K-ary tree of the given depth, scored by prod 1/(rank+1)."""
    nodes = [(1.0, 0, -1)]  # (score, bfs index, parent bfs index)
    frontier = [(0, 1.0)]
    for _ in range(depth):
        nxt = []
        for (idx, sc) in frontier:
            for r in range(K):
                child = len(nodes)
                s = sc / (r + 1)
                nodes.append((s, child, idx))
                nxt.append((child, s))
        frontier = nxt
    order = sorted(range(len(nodes)), key=lambda i: (-nodes[i][0], nodes[i][1]))
    keep = sorted(order[:N], key=lambda i: nodes[i][1])
    renum = {old: new for new, old in enumerate(keep)}
    parent = np.full(len(keep), -1, dtype=np.int32)
    for new, old in enumerate(keep):
        p = nodes[old][2]
        parent[new] = -1 if p < 0 else renum[p]
    return parent


# ------------------------------------------------------------ workloads ----

WORKLOADS = {
    "tiny-linear-b1-k4-v32-f32": dict(B=1, k=4, V=32, dtype="f32", T=1.0, top_p=1.0, seed=0, data_seed=1234),
    "linear-b64-k4-v128256": dict(B=64, k=4, V=128256, dtype="bf16", T=1.0, top_p=1.0, seed=42, data_seed=1235),
    "linear-b256-k8-v128256-t0.7-p0.9": dict(B=256, k=8, V=128256, dtype="bf16", T=0.7, top_p=0.9, seed=42,
                                             data_seed=1236),
    "tree-b32-n60-k4-d5-v128256": dict(B=32, N=60, K=4, depth=5, V=128256, dtype="bf16", T=1.0, top_p=1.0,
                                       seed=42, data_seed=1237),
    "linear-b1024-k3-v129280-h7168": dict(B=1024, k=3, V=129280, H=7168, dtype="bf16", T=1.0, top_p=1.0, seed=42,
                                          data_seed=1238),
}


def linear_logits(B: int, k: int, V: int, dtype: str, data_seed: int, device="cpu", sigma_draft: float = 0.7):
    """(target [B,k+1,V], draft [B,k,V]) per the workload recipe."""
    if dtype == "f32":
        tgt = gaussian((B, k + 1, V), 2.0, data_seed, device)
        drf = (tgt[:, :k].clone() + gaussian((B, k, V), 0.5, data_seed + 1, device))
        return tgt, drf
    tgt = zipf_logits(B * (k + 1), V, data_seed, device).reshape(B, k + 1, V)
    drf = add_noise(tgt[:, :k].contiguous(), sigma_draft, data_seed + 1)
    return tgt, drf


def tree_logits(B: int, N: int, V: int, data_seed: int, device="cpu", sigma_draft: float = 0.7):
    tgt = zipf_logits(B * N, V, data_seed, device).reshape(B, N, V)
    drf = add_noise(tgt, sigma_draft, data_seed + 1)
    return tgt, drf
