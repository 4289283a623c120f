"""Greedy tree/chain verification reproduces autoregressive decoding token for token.

«如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (blog.xiaohack.org/246393),
section 关键突破, reports greedy speculative output bit-identical to plain
autoregressive output over 40 tokens.  Two toy targets check that the oracle
keeps this property:

* a hash model whose next-token logits are a seeded function of the whole
  prefix (checks path selection, the root/bonus convention and A);
* a one-layer random-weight attention model running on the oracle's paged
  attention and commit (checks the tree mask, positions L + depth, and that
  the committed K/V equal those autoregressive decoding would have written).
"""
import hashlib
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_decode_gb300 import synth

V = 64


def _hash_logits(prefix):
    h = hashlib.sha256(np.asarray(prefix, dtype=np.int64).tobytes()).digest()
    return np.random.default_rng(int.from_bytes(h[:8], "little")).standard_normal(V)


def _draw_tree(rng, budget):
    if rng.random() < 0.3:
        return synth.chain_parents(budget)
    return synth.ddtree_parents(rng, budget)[0]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_hash_model_verify_equals_autoregressive(seed):
    rng = np.random.default_rng(seed)
    prompt = list(rng.integers(0, V, size=4))
    n_gen = 48
    ar = list(prompt)
    while len(ar) < len(prompt) + n_gen + 20:
        ar.append(int(np.argmax(_hash_logits(ar))))

    seq = list(prompt)
    steps = 0
    while len(seq) < len(prompt) + n_gen:
        parents = _draw_tree(rng, int(rng.integers(1, 23)))
        n = len(parents)
        paths, _ = oracle.tree_ancestors(parents)
        draft = np.zeros(n, dtype=np.int64)
        draft[0] = seq[-1]
        logits = np.zeros((n, V))
        for j in range(n):
            if j:
                truth = ar[len(seq) + len(paths[j]) - 2]
                draft[j] = truth if rng.random() < 0.75 else int(rng.integers(0, V))
            logits[j] = _hash_logits(seq + [int(draft[i]) for i in paths[j][1:]])
        # duplicate sibling tokens would make "longest" differ from greedy; keep them distinct
        for j in range(1, n):
            while any(draft[i] == draft[j] for i in range(1, j) if parents[i] == parents[j]):
                draft[j] = (draft[j] + 1) % V
        _, lens, pths, toks = oracle.accept([0, n], parents, draft, logits)
        a = int(lens[0])
        _, depth = oracle.tree_ancestors(parents)
        assert 1 <= a <= depth.max() + 1
        seq.extend(toks[0])
        steps += 1
    assert seq == ar[:len(seq)]
    assert steps < n_gen                        # some steps accepted more than one token


class _AttnModel:
    """One attention layer (24 Q / 4 KV heads, d = 256) with random weights."""

    def __init__(self, seed, d_model=32, max_pos=256):
        g = torch.Generator().manual_seed(seed)
        self.emb = torch.randn(V, d_model, generator=g, dtype=torch.float64)
        self.pos = torch.randn(max_pos, d_model, generator=g, dtype=torch.float64)
        self.wq = torch.randn(d_model, 24 * 256, generator=g, dtype=torch.float64) / math.sqrt(d_model)
        self.wk = torch.randn(d_model, 4 * 256, generator=g, dtype=torch.float64) / math.sqrt(d_model)
        self.wv = torch.randn(d_model, 4 * 256, generator=g, dtype=torch.float64) / math.sqrt(d_model)
        self.wo = torch.randn(24 * 256, V, generator=g, dtype=torch.float64) / 8.0

    def qkv(self, tokens, positions):
        x = self.emb[list(tokens)] + self.pos[list(positions)]
        bf = lambda t: t.to(torch.bfloat16).to(torch.float64).numpy()   # stored as bf16
        return (bf(x @ self.wq).reshape(-1, 24, 256), bf(x @ self.wk).reshape(-1, 4, 256),
                bf(x @ self.wv).reshape(-1, 4, 256))

    def logits(self, o):
        return (torch.from_numpy(o.reshape(o.shape[0], -1)) @ self.wo).numpy()


class _Cache:
    def __init__(self, rng, pages=24):
        self.table = rng.permutation(pages).astype(np.int32)[None, :]
        self.k = [np.zeros((pages, 4, 16, 256))]
        self.v = [np.zeros((pages, 4, 16, 256))]
        self.ctx = np.array([0])

    def step(self, model, tokens_of_nodes, parents):
        """One verify forward; returns per-node logits and the tree's keys."""
        _, depth = oracle.tree_ancestors(parents)
        L = int(self.ctx[0])
        q, kn, vn = model.qkv(tokens_of_nodes, [L + int(d) for d in depth])
        o, _ = oracle.verify_attention(q, self.k[0], self.v[0], kn, vn, self.table, self.ctx,
                                       [0, len(parents)], parents)
        return model.logits(o), kn, vn

    def commit(self, kn, vn, a, path):
        self.k, self.v, self.ctx = oracle.kv_commit(self.k, self.v, [kn], [vn], self.table, self.ctx,
                                                    [0, len(kn)], [a], [path])


@pytest.mark.parametrize("seed", [0, 1])
def test_attention_model_verify_equals_autoregressive(seed):
    rng = np.random.default_rng(100 + seed)
    model = _AttnModel(seed)
    prompt = [int(x) for x in rng.integers(0, V, size=5)]
    n_gen = 40

    # autoregressive: every step is a one-node block (the root)
    ar_cache = _Cache(np.random.default_rng(seed))
    ar = list(prompt)
    for i in range(len(prompt) - 1):                        # prefill, teacher-forced
        _, kn, vn = ar_cache.step(model, [prompt[i]], np.array([-1]))
        ar_cache.commit(kn, vn, 1, [0])
    while len(ar) < len(prompt) + n_gen + 17:
        lg, kn, vn = ar_cache.step(model, [ar[-1]], np.array([-1]))
        ar_cache.commit(kn, vn, 1, [0])
        ar.append(int(np.argmax(lg[0])))

    cache = _Cache(np.random.default_rng(seed))
    for i in range(len(prompt) - 1):
        _, kn, vn = cache.step(model, [prompt[i]], np.array([-1]))
        cache.commit(kn, vn, 1, [0])
    seq = list(prompt)
    steps = 0
    while len(seq) < len(prompt) + n_gen:
        parents = _draw_tree(rng, int(rng.integers(1, 12)))
        paths, _ = oracle.tree_ancestors(parents)
        draft = [seq[-1]]
        for j in range(1, len(parents)):
            truth = ar[len(seq) + len(paths[j]) - 2]
            tok = truth if (rng.random() < 0.8) else int(rng.integers(0, V))
            while any(draft[i] == tok for i in range(1, j) if parents[i] == parents[j]):
                tok = (tok + 1) % V
            draft.append(tok)
        lg, kn, vn = cache.step(model, draft, parents)
        _, lens, pths, toks = oracle.accept([0, len(parents)], parents, draft, lg)
        cache.commit(kn, vn, int(lens[0]), pths[0])
        seq.extend(toks[0])
        steps += 1
    assert seq == ar[:len(seq)]
    assert steps < n_gen
    # the committed cache equals the autoregressive one position by position
    n = int(cache.ctx[0])
    np.testing.assert_array_equal(oracle.gather_context(cache.k[0], cache.table[0], n),
                                  oracle.gather_context(ar_cache.k[0], ar_cache.table[0], n))
