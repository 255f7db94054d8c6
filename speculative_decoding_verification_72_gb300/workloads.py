"""Seeded synthetic inputs shaped like the pages' verification workloads.

This module only draws inputs. It holds none of the verification arithmetic,
so both the CUDA path's tests and the CPU oracle's tests can take their inputs
from it. Random numbers come from torch generators (CPU or CUDA, as asked);
tree shapes come from a NumPy generator on the host.

Workloads (no dataset, prompt or weight is reproduced: only vocabulary sizes,
draft lengths and tree shapes are taken from the pages):
  toy_chain        B=4, K=4, V=32 fp32 logits ~ N(0, 2^2); draft q is the mix
                   0.8 p + 0.2 softmax(N(0, 2^2)), passed as log q; drafts
                   sampled from q (spec-decode README, toy draft with agreement).
  greedy_chain     bf16 logits ~ N(0, 3^2); each draft equals its row's argmax
                   with probability p_match, else a uniformly random other id
                   (Llama-3 vocabulary 128256 with K=5, the chain of the
                   nanospec README; GPT-2 vocabulary 50257 with K+1=4096 rows,
                   the spec100m README's tokens per step).
  stochastic_chain fp32 target logits ~ N(0, 3^2); draft logits = target +
                   N(0, 1^2); drafts sampled from softmax(draft / T) (Qwen
                   vocabulary 151936, K=4, as in mini-sglang PR #134's K=4).
  eagle_tree       EAGLE-3-style tree, depth 5 and top-4 expansion pruned to
                   64 nodes including the root (nanospec README, tree config),
                   bf16 logits ~ N(0, 3^2).
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch


@dataclass
class ChainInputs:
    target: torch.Tensor                  # [B, K+1, V] bf16 or fp32
    draft_tokens: torch.Tensor            # [B, K] int32
    uniforms: torch.Tensor                # [B, K+1] fp32 in [0, 1)
    draft_logits: Optional[torch.Tensor] = None   # [B, K, V] or None
    temperature: float = 1.0


@dataclass
class TreeInputs:
    target: torch.Tensor                  # [B, N, V]
    node_tokens: torch.Tensor             # [B, N] int32 (node 0 = root)
    parents: torch.Tensor                 # [B, N] int32 (parents[:, 0] = -1)
    uniforms: torch.Tensor                # [B, N] fp32
    max_depth: int = 5


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal_logits(B, R, V, std, dtype, device, g, chunk_rows=4096):
    out = torch.empty((B, R, V), dtype=dtype, device=device)
    flat = out.view(B * R, V)
    for r0 in range(0, B * R, chunk_rows):
        r1 = min(B * R, r0 + chunk_rows)
        blk = torch.randn((r1 - r0, V), generator=g, device=device, dtype=torch.float32)
        flat[r0:r1] = (blk * std).to(dtype)
    return out


def _other_ids(argmax, V, g, device):
    if V == 1:
        return torch.zeros_like(argmax)
    r = torch.randint(0, V - 1, argmax.shape, generator=g, device=device, dtype=torch.int64)
    return r + (r >= argmax).to(torch.int64)


def greedy_chain(B, K, V, dtype=torch.bfloat16, std=3.0, p_match=0.8, seed=7201,
                 device="cpu"):
    g = _gen(device, seed)
    target = _normal_logits(B, K + 1, V, std, dtype, device, g)
    am = torch.argmax(target[:, :K, :], dim=-1).to(torch.int64) if K > 0 else \
        torch.zeros((B, 0), dtype=torch.int64, device=device)
    coin = torch.rand((B, K), generator=g, device=device) < p_match
    drafts = torch.where(coin, am, _other_ids(am, V, g, device))
    uniforms = torch.rand((B, K + 1), generator=g, device=device, dtype=torch.float32)
    return ChainInputs(target=target, draft_tokens=drafts.to(torch.int32).contiguous(),
                       uniforms=uniforms)


def stochastic_chain(B, K, V, dtype=torch.float32, std=3.0, noise=1.0, temperature=1.0,
                     seed=7202, device="cpu"):
    g = _gen(device, seed)
    target = _normal_logits(B, K + 1, V, std, dtype, device, g)
    draft = torch.empty((B, K, V), dtype=dtype, device=device)
    for b in range(B):
        eps = torch.randn((K, V), generator=g, device=device, dtype=torch.float32)
        draft[b] = (target[b, :K].float() + noise * eps).to(dtype)
    probs = torch.softmax(draft.float().view(B * K, V) / temperature, dim=-1)
    drafts = torch.multinomial(probs, 1, generator=g).view(B, K) if K > 0 else \
        torch.zeros((B, 0), dtype=torch.int64, device=device)
    uniforms = torch.rand((B, K + 1), generator=g, device=device, dtype=torch.float32)
    return ChainInputs(target=target, draft_tokens=drafts.to(torch.int32).contiguous(),
                       uniforms=uniforms, draft_logits=draft, temperature=temperature)


def toy_chain(B=4, K=4, V=32, std=2.0, agreement=0.8, seed=7200, device="cpu"):
    """Target N(0, 2^2) fp32; draft probabilities 0.8 p + 0.2 softmax(N(0, 2^2))."""
    g = _gen(device, seed)
    target = _normal_logits(B, K + 1, V, std, torch.float32, device, g)
    other = torch.randn((B, K, V), generator=g, device=device) * std
    q = agreement * torch.softmax(target[:, :K].double(), -1) + \
        (1 - agreement) * torch.softmax(other.double(), -1)
    draft_logits = torch.log(q).float()
    drafts = torch.multinomial(q.view(B * K, V).float(), 1, generator=g).view(B, K)
    uniforms = torch.rand((B, K + 1), generator=g, device=device, dtype=torch.float32)
    return ChainInputs(target=target, draft_tokens=drafts.to(torch.int32).contiguous(),
                       uniforms=uniforms, draft_logits=draft_logits, temperature=1.0)


def toy_greedy_drafts(target, p_match=0.8, seed=7210):
    """Greedy drafts for an existing [B, K+1, V] target: argmax w.p. p_match."""
    B, R, V = target.shape
    K = R - 1
    g = _gen(target.device, seed)
    am = torch.argmax(target[:, :K], dim=-1).to(torch.int64)
    coin = torch.rand((B, K), generator=g, device=target.device) < p_match
    return torch.where(coin, am, _other_ids(am, V, g, target.device)).to(torch.int32)


# ------------------------------------------------------------------ trees

def tree_shape(rng, depth=5, topk=4, n_nodes=64):
    """Parent array (BFS order, parents[0] = -1) of an EAGLE-3-style tree.

    Level 1 is topk children of the root; every later level expands the topk
    best nodes of the level above (by cumulative score; each child adds a
    seeded -Exp(1) increment, so scores fall along a path) into topk children
    each. The n_nodes - 1 best candidates are kept (ancestor-closed, since a
    parent always outscores its child; ties go to the earlier candidate) and
    renumbered in BFS order, siblings in descending score order.
    """
    cands = []   # (level, score, parent_candidate, index)
    level_nodes = [(-1, 0.0)]   # (candidate index or -1 for root, score)
    for level in range(1, depth + 1):
        if level == 1:
            parents = level_nodes
        else:
            ranked = sorted(level_nodes, key=lambda t: (-t[1], t[0]))
            parents = ranked[:topk]
        nxt = []
        for (pc, ps) in parents:
            for _ in range(topk):
                s = ps - float(rng.exponential(1.0))
                idx = len(cands)
                cands.append((level, s, pc, idx))
                nxt.append((idx, s))
        level_nodes = nxt
    keep = sorted(cands, key=lambda c: (-c[1], c[3]))[: n_nodes - 1]
    keep_set = {c[3] for c in keep}
    for c in keep:   # ancestor closure holds because scores fall along a path
        assert c[2] == -1 or c[2] in keep_set
    order = sorted(keep, key=lambda c: (c[0], -c[1], c[3]))
    new_index = {c[3]: i + 1 for i, c in enumerate(order)}
    parents = np.full(len(order) + 1, -1, dtype=np.int64)
    for c in order:
        parents[new_index[c[3]]] = 0 if c[2] == -1 else new_index[c[2]]
    return parents


def eagle_tree(B, V, n_nodes=64, depth=5, topk=4, dtype=torch.bfloat16, std=3.0,
               p_first_is_argmax=0.8, seed=7203, device="cpu"):
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    target = _normal_logits(B, n_nodes, V, std, dtype, device, g)
    am = torch.argmax(target, dim=-1).cpu().numpy()          # [B, N]
    parents = np.zeros((B, n_nodes), dtype=np.int64)
    tokens = np.zeros((B, n_nodes), dtype=np.int64)
    for b in range(B):
        par = tree_shape(rng, depth, topk, n_nodes)
        parents[b] = par
        for n in range(n_nodes):
            kids = [c for c in range(1, n_nodes) if par[c] == n]
            used = set()
            for j, c in enumerate(kids):
                if j == 0 and rng.random() < p_first_is_argmax:
                    t = int(am[b, n])
                else:
                    while True:
                        t = int(rng.integers(0, V))
                        if t != am[b, n] and t not in used:
                            break
                used.add(t)
                tokens[b, c] = t
    uniforms = torch.rand((B, n_nodes), generator=g, device=device, dtype=torch.float32)
    return TreeInputs(target=target,
                      node_tokens=torch.from_numpy(tokens).to(torch.int32).to(device),
                      parents=torch.from_numpy(parents).to(torch.int32).to(device),
                      uniforms=uniforms, max_depth=depth)


def draft_tree_rows(B, V, depth=5, topk=4, dtype=torch.bfloat16, std=3.0, seed=7205, device="cpu"):
    """Rank-ordered draft rows for tree construction: [B, 1 + (depth - 1) * topk, V]
    logits N(0, std^2) (row 0 the root's, then topk rows per later level)."""
    g = _gen(device, seed)
    return _normal_logits(B, 1 + (depth - 1) * topk, V, std, dtype, device, g)
