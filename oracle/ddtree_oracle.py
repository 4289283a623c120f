"""Oracle for the draft-tree (DDTree) construction that precedes the verify step.

TEST INFRASTRUCTURE ONLY.  Plain, slow CPU reference; only the tests, the smoke
check and the bench's CPU-baseline leg may import it.  It shares no code with
the CUDA path and imports nothing from the product package.

Source: «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (S5).
[从自回归到 DDTree]: a draft block of 16 positions is expanded into a token tree
of `budget` nodes that the target verifies in one forward pass.  [关键突破]:
the tree is built from the draft's per-position top-K (K = 32 -> 8), with a
chain pre-seed; a top-K list in the wrong order (worst candidate first) sends
the worst token to the root's child and every step accepts 1.

Readings where the page is silent (each is listed in the design notes):

* each position's candidates are its top-K tokens by draft logit (ties: the
  smaller token id first), scored by log-probability logit - logsumexp(row);
* a node at depth d >= 1 holds a candidate of position d - 1; its score is the
  sum of the log-probabilities on its root path (the root scores 0);
* chain pre-seed: the rank-0 chain (the draft's greedy continuation) up to
  depth min(positions, budget) is inserted first;
* the rest is best-first: a candidate heap holds, for every inserted node, its
  first child (rank 0, one position deeper) and its next sibling (rank + 1,
  same parent); the highest score is inserted next, ties to the candidate
  created first; this enumerates prefixes in score order because log-probs
  are <= 0 and a position's candidates are sorted;
* nodes are numbered in insertion order (root 0), so parent[j] < j.
Everything is float64.
"""
from __future__ import annotations

import heapq

import numpy as np


def topk_first(row, k: int) -> np.ndarray:
    """Indices of the k largest values, largest first; equal values: smaller index first."""
    x = np.asarray(row, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN in draft logits")
    order = np.lexsort((np.arange(x.size), -x))     # primary: value descending; then index ascending
    return order[:k]


def logsumexp(row) -> float:
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    return float(m + np.log(np.exp(x - m).sum()))


def candidates(draft_logits, k: int):
    """Per position: (tokens [k], log-probabilities [k]) of the top-k candidates."""
    toks, lps = [], []
    for row in np.asarray(draft_logits):
        idx = topk_first(row, k)
        toks.append(idx.astype(np.int64))
        lps.append(np.asarray(row, dtype=np.float64)[idx] - logsumexp(row))
    return np.stack(toks), np.stack(lps)


def build_tree(cand_tokens, cand_logprobs, budget: int, root_token: int):
    """Best-first tree of 1 + budget nodes over the candidates (see the module notes).

    Returns (parents [n], tokens [n], scores [n], margin): `margin` is the smallest
    score gap between the candidate inserted and the best lower-scored one left
    behind, over all best-first decisions (inf when no choice was contested).
    """
    positions, k = cand_tokens.shape
    parents, tokens, scores = [-1], [int(root_token)], [0.0]
    depth_of, rank_of = [0], [0]
    chain = min(positions, budget)
    for d in range(1, chain + 1):                       # the chain pre-seed
        parents.append(d - 1)
        tokens.append(int(cand_tokens[d - 1, 0]))
        scores.append(scores[-1] + float(cand_logprobs[d - 1, 0]))
        depth_of.append(d)
        rank_of.append(0)
    heap: list = []
    seq = 0

    def push(parent: int, depth: int, rank: int):
        nonlocal seq
        if depth > positions or rank >= k:
            return
        s = scores[parent] + float(cand_logprobs[depth - 1, rank])
        heapq.heappush(heap, (-s, seq, parent, depth, rank))
        seq += 1

    for d in range(0, chain):                           # second-best child of every chain node with a
        push(d, d + 1, 1)                               # chain child (its best child is in the chain)
    push(chain, chain + 1, 0)                           # and the chain's continuation below its end
    margin = float("inf")
    while len(parents) < 1 + budget and heap:
        neg, _, par, dep, rk = heapq.heappop(heap)
        lower = [h[0] for h in heap if h[0] > neg]      # candidates left behind with a lower score
        if lower:                                       # (equal scores are ordered by creation on
            margin = min(margin, min(lower) - neg)       # any hardware, so they are not a contest)
        node = len(parents)
        parents.append(par)
        tokens.append(int(cand_tokens[dep - 1, rk]))
        scores.append(-neg)
        depth_of.append(dep)
        rank_of.append(rk)
        push(node, dep + 1, 0)                          # its first child
        push(par, dep, rk + 1)                          # its next sibling
    return (np.asarray(parents, dtype=np.int64), np.asarray(tokens, dtype=np.int64),
            np.asarray(scores, dtype=np.float64), margin)


def ddtree(draft_logits, k: int, budget: int, root_token: int):
    """Candidates then tree for one sequence: draft_logits [positions, V]."""
    ct, cl = candidates(draft_logits, k)
    return build_tree(ct, cl, budget, root_token)
