"""Oracle for the target-model verify step of speculative decoding.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, CPU reference that
the CUDA path is checked against.  Only the tests, the smoke check and the
bench's CPU-baseline leg may import it.  It shares no code with the CUDA path,
and it neither imports the product package nor is imported by it.

Everything is computed in float64 from the bf16-decoded inputs (the caller
passes float arrays holding exactly the bf16 values).  Library primitives used
as steps: numpy matrix-vector products, ``max``, ``exp``, ``log``, ``sum``.

Sources (page titles; sections in brackets):

* [S5] «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍»
  (blog.xiaohack.org/246393).  [为什么我们要做这个测试]: 24 Q heads, 4 KV heads,
  head dim 256.  [架构设计]: greedy verify, draft block 16.  [从自回归到 DDTree]:
  accept length (AL) = tokens accepted per verify step.  [关键突破]: a tree
  node sees its parent chain (siblings gather along the parent chain);
  the verify logits buffer holds vocab x (budget + 1) rows; greedy DFlash output
  is bit-identical to autoregressive output; a reversed top-K made every step
  accept exactly 1.
* [S1] «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图»
  (xdnf.cn/news/337238).  [2]: paged KV cache, 16 tokens per page.  [4]: all
  verify slots draw physical pages from one pool.  [5.3]: the causal mask of a
  multi-token draft must let draft j see exactly the context plus drafts 0..j.
* [S3] «Qwen3.8-27B 部署技术报告» (FlintyLemming): chain drafts of 4 (MTP) and 8
  (DFlash2), temperature 0 in every test.

Readings where the pages are silent (each is also listed in the design notes):

* softmax scale 1/sqrt(256) = 1/16;
* query head h reads KV head h // 6 (contiguous groups of 6);
* node 0 of each draft block is the root, i.e. the last emitted token, whose
  K/V is not cached yet; it is a query, and it is committed with the accepted
  path, so a step commits A tokens;
* key order for node j: context positions 0..L-1, then draft nodes on j's root
  path in increasing index (j included);
* argmax ties go to the smallest index; -0.0 equals +0.0; NaN is rejected;
* among accepted root paths of maximal length, ties go to the
  lexicographically smallest sequence of node indices;
* A = accepted drafts + 1 (root counts), so an all-rejected step gives A = 1;
* sliding window W [S5 补充测试: attention over the most recent 2,048 KV
  positions only]: node j sits at position L + depth(j), and a key at position
  t is visible to it when t > L + depth(j) - W (the W most recent positions,
  its own included); a draft ancestor n is at position L + depth(n).
"""
from __future__ import annotations

import numpy as np

PAGE = 16          # tokens per KV page [S1 §2]
H_Q = 24           # query heads [S5 为什么我们要做这个测试]
H_KV = 4           # KV heads
GROUP = H_Q // H_KV
HEAD_DIM = 256
SCALE = 1.0 / 16.0  # 1/sqrt(HEAD_DIM)


# ---------------------------------------------------------------- tree mask

def tree_ancestors(parents) -> tuple[list[list[int]], np.ndarray]:
    """Validate a parent array and return, per node, its root path and depth.

    ``parents[0] == -1`` (the root) and ``0 <= parents[j] < j`` otherwise.
    The root path of j lists the nodes from the root down to j (j included) in
    increasing index order; these are the draft keys node j may attend to
    [S5 关键突破: siblings follow their own parent chain].
    """
    par = [int(x) for x in np.asarray(parents).reshape(-1)]
    if len(par) == 0:
        raise ValueError("empty draft block")
    if par[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for j in range(1, len(par)):
        if not (0 <= par[j] < j):
            raise ValueError(f"parent of node {j} is {par[j]}; need 0 <= parent < {j}")
    paths: list[list[int]] = []
    depth = np.zeros(len(par), dtype=np.int64)
    for j in range(len(par)):
        chain = []
        u = j
        while u != -1:
            chain.append(u)
            u = par[u]
        chain.reverse()
        paths.append(chain)
        depth[j] = len(chain) - 1
    return paths, depth


# ---------------------------------------------------------------- attention

def gather_context(cache, table_row, ctx_len: int, head: int | None = None) -> np.ndarray:
    """Token p of a sequence lives in page ``table_row[p // 16]``, slot ``p % 16``.

    ``cache`` is [pool_pages, H_KV, 16, D]; returns [ctx_len, H_KV, D] float64,
    or [ctx_len, D] for one KV ``head``.
    """
    cache = np.asarray(cache)
    table_row = np.asarray(table_row)
    pos = np.arange(ctx_len)
    pages = table_row[pos // PAGE].astype(np.int64)
    if ctx_len and (pages.min() < 0 or pages.max() >= cache.shape[0]):
        raise ValueError("page table entry outside the pool")
    if head is None:
        return np.asarray(cache[pages, :, pos % PAGE, :], dtype=np.float64)
    return np.asarray(cache[pages, head, pos % PAGE, :], dtype=np.float64)


def attend(qv, keys, values, visible) -> tuple[np.ndarray, float]:
    """Masked softmax attention of one query vector.

    s_i = (q . k_i) / 16 for visible keys (masked keys get s_i = -inf, so their
    weight exp(-inf) is exactly 0);  m = max_i s_i;
    o = sum_i exp(s_i - m) v_i / sum_i exp(s_i - m);  lse = m + log sum_i exp(s_i - m).
    """
    s = (keys @ np.asarray(qv, dtype=np.float64)) * SCALE
    s = np.where(visible, s, -np.inf)
    m = s.max()
    w = np.exp(s - m)
    denom = w.sum()
    o = (w @ values) / denom
    return o, float(m + np.log(denom))


def verify_attention(q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, q_indptr, parents,
                     samples=None, window=None):
    """Tree/causal-masked grouped-query attention of one layer.

    q [sumN, 24, D]; k_cache/v_cache [P, 4, 16, D]; k_new/v_new [sumN, 4, D];
    page_table [B, max_pages]; ctx_lens [B]; q_indptr [B+1]; parents [sumN]
    (per-sequence local ids).  Query (node j, head h) of sequence b attends to
    all L_b context tokens and to the draft nodes on j's root path, reading KV
    head h // 6.  Keys are laid out as [context 0..L-1, draft nodes 0..N-1].

    Returns (o [sumN, 24, D], lse [sumN, 24]) in float64.  With ``samples`` (a
    list of (row, head) pairs) only those entries are computed and the result
    is (o [S, D], lse [S]).  With ``window`` W >= 1 each query sees only the
    keys at its W most recent positions (node j at position L + depth(j)
    [S5 补充测试]); None or 0 means the whole context.
    """
    q = np.asarray(q)
    indptr = np.asarray(q_indptr)
    batch = len(indptr) - 1
    row_seq = np.repeat(np.arange(batch), np.diff(indptr))
    if samples is None:
        want = [(r, h) for r in range(int(indptr[-1])) for h in range(H_Q)]
    else:
        want = [(int(r), int(h)) for r, h in samples]
    by_seq_head: dict[tuple[int, int], list[int]] = {}
    for i, (r, h) in enumerate(want):
        by_seq_head.setdefault((int(row_seq[r]), h // GROUP), []).append(i)
    o_out = np.zeros((len(want), q.shape[-1]), dtype=np.float64)
    lse_out = np.zeros(len(want), dtype=np.float64)
    for (b, g), items in sorted(by_seq_head.items()):
        lo, hi = int(indptr[b]), int(indptr[b + 1])
        paths, depth = tree_ancestors(np.asarray(parents)[lo:hi])
        L = int(np.asarray(ctx_lens)[b])
        row = np.asarray(page_table)[b]
        keys = np.concatenate([gather_context(k_cache, row, L, g),
                               np.asarray(k_new, dtype=np.float64)[lo:hi, g, :]])
        vals = np.concatenate([gather_context(v_cache, row, L, g),
                               np.asarray(v_new, dtype=np.float64)[lo:hi, g, :]])
        for i in items:
            r, h = want[i]
            visible = np.zeros(L + hi - lo, dtype=bool)
            if window:
                pos = L + int(depth[r - lo])                 # this query's position
                first = max(0, pos - int(window) + 1)        # oldest visible position
                visible[first:L] = True
                visible[[L + n for n in paths[r - lo] if L + int(depth[n]) >= first]] = True
            else:
                visible[:L] = True
                visible[[L + n for n in paths[r - lo]]] = True
            o_out[i], lse_out[i] = attend(q[r, h, :], keys, vals, visible)
    if samples is not None:
        return o_out, lse_out
    n = int(indptr[-1])
    return o_out.reshape(n, H_Q, -1), lse_out.reshape(n, H_Q)


# ---------------------------------------------------------------- argmax

def argmax_first(logits) -> np.ndarray:
    """Per row, the smallest index attaining the row maximum (greedy decoding).

    Rows must be finite (NaN is rejected).  -0.0 and +0.0 compare equal.
    """
    x = np.asarray(logits)
    if x.ndim == 1:
        x = x[None, :]
    if np.isnan(x).any():
        raise ValueError("NaN in logits")
    out = np.empty(x.shape[0], dtype=np.int64)
    for r in range(x.shape[0]):
        row = x[r]
        out[r] = int(np.flatnonzero(row == row.max())[0])
    return out


# ---------------------------------------------------------------- accept

def root_to_leaf_paths(parents) -> list[list[int]]:
    """Every path from the root to a node without children."""
    par = [int(x) for x in np.asarray(parents)]
    children = [[] for _ in par]
    for j in range(1, len(par)):
        children[par[j]].append(j)
    out: list[list[int]] = []
    stack = [[0]]
    while stack:
        path = stack.pop()
        kids = children[path[-1]]
        if not kids:
            out.append(path)
        for c in kids:
            stack.append(path + [c])
    return out


def accept_bruteforce(parents, draft, t) -> tuple[int, list[int], list[int]]:
    """Greedy acceptance of one sequence's draft tree, by enumerating paths.

    Along a root-to-leaf path the accepted prefix keeps extending while the
    next node's draft token equals the target's greedy token at its parent
    [S5 架构设计: greedy verify].  The longest accepted prefix over all paths
    wins (ties: lexicographically smallest node sequence).  A = its length in
    nodes (root included) [S5 从自回归到 DDTree: AL]; the emitted tokens are the
    accepted drafts followed by one bonus token, the target's greedy token at
    the last accepted node.

    Returns (A, path node ids [A], emitted tokens [A]).
    """
    tree_ancestors(parents)                      # validation
    draft = [int(x) for x in np.asarray(draft)]
    t = [int(x) for x in np.asarray(t)]
    best: list[int] | None = None
    for path in root_to_leaf_paths(parents):
        k = 1
        while k < len(path) and draft[path[k]] == t[path[k - 1]]:
            k += 1
        prefix = path[:k]
        if best is None or len(prefix) > len(best) or (len(prefix) == len(best) and prefix < best):
            best = prefix
    assert best is not None
    tokens = [draft[n] for n in best[1:]] + [t[best[-1]]]
    return len(best), best, tokens


def accept(q_indptr, parents, draft_tokens, logits):
    """Argmax of every logits row, then path selection per sequence.

    ``logits`` has one row per draft node, root included, i.e. budget + 1 rows
    per sequence [S5 关键突破: verify_logits_buf].
    Returns (t [sumN], accept_len [B], paths (list of lists), tokens (list of lists)).
    """
    indptr = np.asarray(q_indptr)
    logits = np.asarray(logits)
    if logits.shape[0] != int(indptr[-1]):
        raise ValueError("need one logits row per draft node (budget + 1 per sequence)")
    t = argmax_first(logits)
    lens, paths, toks = [], [], []
    for b in range(len(indptr) - 1):
        lo, hi = int(indptr[b]), int(indptr[b + 1])
        a, path, tok = accept_bruteforce(np.asarray(parents)[lo:hi], np.asarray(draft_tokens)[lo:hi],
                                         t[lo:hi])
        lens.append(a)
        paths.append(path)
        toks.append(tok)
    return t, np.asarray(lens, dtype=np.int64), paths, toks


# ---------------------------------------------------------------- commit

def kv_commit(k_caches, v_caches, k_news, v_news, page_table, ctx_lens, q_indptr, accept_len, paths):
    """Append the accepted nodes' K/V to each sequence's cache, for every layer.

    Accepted node path[i] (i < A) goes to position L + i: page
    ``table[(L + i) // 16]``, slot ``(L + i) % 16`` [S1 §2, §4]; rejected nodes are
    never written.  Works on copies of the caches (arrays of any dtype; bytes
    are copied unchanged).  Returns (new k caches, new v caches, new ctx_lens).
    """
    indptr = np.asarray(q_indptr)
    table = np.asarray(page_table)
    ks = [np.array(c, copy=True) for c in k_caches]
    vs = [np.array(c, copy=True) for c in v_caches]
    new_ctx = np.asarray(ctx_lens, dtype=np.int64).copy()
    for b in range(len(indptr) - 1):
        L = int(new_ctx[b])
        for i in range(int(accept_len[b])):
            pos = L + i
            page = int(table[b, pos // PAGE])
            if not (0 <= page < ks[0].shape[0]):
                raise ValueError("commit target outside the page pool")
            src = int(indptr[b]) + int(paths[b][i])
            for layer in range(len(ks)):
                ks[layer][page, :, pos % PAGE, :] = np.asarray(k_news[layer])[src]
                vs[layer][page, :, pos % PAGE, :] = np.asarray(v_news[layer])[src]
        new_ctx[b] = L + int(accept_len[b])
    return ks, vs, new_ctx
