"""Pins for the oracle's argmax, path selection and commit.

Greedy verification and the accept length come from «如何在单张 RTX 3090 上让
Qwen3.5-27B token 生成速度提升 6 倍» (blog.xiaohack.org/246393): 架构设计 (greedy
verify), 从自回归到 DDTree (AL), 关键突破 (parent-chain siblings; budget+1 logits
rows; greedy output bit-identical to autoregressive decoding; a reversed
top-K gave accept = 1 on every step).
"""
import json
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_verify_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")


# ------------------------------------------------------------------ argmax

def test_argmax_matches_numpy_first_occurrence():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((17, 5003)).astype(np.float32)
    x[3, 100] = x[3, 4000] = 9.0          # tie: first index wins
    x[5] = 1.0                             # all equal: index 0
    np.testing.assert_array_equal(oracle.argmax_first(x), np.argmax(x, axis=1))


def test_argmax_ties_and_signed_zero():
    assert oracle.argmax_first(np.array([1.0, 3.0, 2.0, 3.0]))[0] == 1
    assert oracle.argmax_first(np.array([-0.0, 0.0, -1.0]))[0] == 0
    assert oracle.argmax_first(np.array([-1.0, 0.0, -0.0]))[0] == 1
    assert oracle.argmax_first(np.array([-np.inf, -np.inf]))[0] == 0
    assert oracle.argmax_first(np.array([-5.0, np.inf, np.inf]))[0] == 1


def test_argmax_rejects_nan():
    with pytest.raises(ValueError):
        oracle.argmax_first(np.array([0.0, np.nan]))


# ------------------------------------------------------------------ accept

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_accept_golden(case):
    a, path, toks = oracle.accept_bruteforce(case["parents"], case["draft"], case["t"])
    assert (a, path, toks) == (case["accept_len"], case["path"], case["tokens"])


def _greedy_walk(parents, draft, t):
    """Follow, from the root, the lowest-index child carrying the parent's greedy token."""
    cur, path = 0, [0]
    while True:
        nxt = [j for j in range(1, len(parents)) if parents[j] == cur and draft[j] == t[cur]]
        if not nxt:
            return path
        cur = nxt[0]
        path.append(cur)


@pytest.mark.parametrize("seed", range(40))
def test_bruteforce_equals_greedy_walk_with_distinct_siblings(seed):
    rng = np.random.default_rng(seed)
    par, spine = synth.ddtree_parents(rng, int(rng.integers(1, 40)))
    t = rng.integers(0, 50, size=len(par))
    draft = synth.plant_drafts(rng, par, t, 50, 0.7, planted=np.ones(len(par), bool))
    a, path, toks = oracle.accept_bruteforce(par, draft, t)
    assert path == _greedy_walk(par, draft, t)
    _, depth = oracle.tree_ancestors(par)
    assert 1 <= a <= depth.max() + 1
    assert toks[-1] == t[path[-1]]
    assert toks[:-1] == [int(draft[n]) for n in path[1:]]


def test_all_rejected_is_one_autoregressive_step():
    rng = np.random.default_rng(7)
    par = synth.ddtree_parents(rng, 22)[0]
    logits = rng.standard_normal((23, 300))
    t = np.argmax(logits, axis=1)
    draft = np.array([(int(t[max(p, 0)]) + 1) % 300 for p in par])
    tt, lens, paths, toks = oracle.accept([0, 23], par, draft, logits)
    assert lens[0] == 1 and paths[0] == [0] and toks[0] == [int(np.argmax(logits[0]))]


def test_logits_need_budget_plus_one_rows():
    with pytest.raises(ValueError):
        oracle.accept([0, 5], synth.chain_parents(4), np.zeros(5, int), np.zeros((4, 10)))


def test_mean_accept_length_of_planted_chain():
    # With each chain draft accepted independently with probability p, the
    # expected accept length (root counted) is (1 - p^(K+1)) / (1 - p).
    rng = np.random.default_rng(123)
    k, p, trials = 4, 0.8, 4000
    par = synth.chain_parents(k)
    total = 0
    for _ in range(trials):
        t = rng.integers(0, 1000, size=k + 1)
        draft = synth.plant_drafts(rng, par, t, 1000, p)
        total += oracle.accept_bruteforce(par, draft, t)[0]
    expect = (1 - p ** (k + 1)) / (1 - p)
    assert abs(total / trials - expect) < 4 * 1.6 / np.sqrt(trials)


# ------------------------------------------------------------------ commit

def _rand_cache(rng, pages):
    return rng.integers(0, 1 << 16, size=(pages, 4, 16, 256), dtype=np.uint16)


def test_commit_writes_accepted_slots_only():
    rng = np.random.default_rng(1)
    w = synth.make_structure(3, [30, 0, 47], [synth.chain_parents(4),
                                              synth.ddtree_parents(rng, 9)[0],
                                              synth.chain_parents(2)], 9, 100, [0.6] * 3, spare_pages=4)
    layers = 2
    kc = [_rand_cache(rng, w.num_pool_pages) for _ in range(layers)]
    vc = [_rand_cache(rng, w.num_pool_pages) for _ in range(layers)]
    kn = [rng.integers(0, 1 << 16, size=(w.total_nodes, 4, 256), dtype=np.uint16) for _ in range(layers)]
    vn = [rng.integers(0, 1 << 16, size=(w.total_nodes, 4, 256), dtype=np.uint16) for _ in range(layers)]
    lens = np.array([5, 3, 1])
    paths = [[0, 1, 2, 3, 4], [0, 1, 2], [0]]
    ks, vs, new_ctx = oracle.kv_commit(kc, vc, kn, vn, w.page_table, w.ctx_lens, w.q_indptr, lens, paths)
    assert list(new_ctx) == [35, 3, 48]
    for layer in range(layers):
        touched = np.zeros((w.num_pool_pages, 16), dtype=bool)
        for b in range(3):
            for i, node in enumerate(paths[b]):
                pos = int(w.ctx_lens[b]) + i
                page = int(w.page_table[b, pos // 16])
                touched[page, pos % 16] = True
                src = int(w.q_indptr[b]) + node
                np.testing.assert_array_equal(ks[layer][page, :, pos % 16], kn[layer][src])
                np.testing.assert_array_equal(vs[layer][page, :, pos % 16], vn[layer][src])
        untouched = ~touched
        np.testing.assert_array_equal(ks[layer].transpose(0, 2, 1, 3)[untouched],
                                      kc[layer].transpose(0, 2, 1, 3)[untouched])
        np.testing.assert_array_equal(vs[layer].transpose(0, 2, 1, 3)[untouched],
                                      vc[layer].transpose(0, 2, 1, 3)[untouched])


def test_commit_of_full_chain_is_contiguous_append():
    rng = np.random.default_rng(2)
    w = synth.make_structure(1, [29], [synth.chain_parents(8)], 3, 100, [0.9])
    kc = [_rand_cache(rng, w.num_pool_pages)]
    kn = [rng.integers(0, 1 << 16, size=(9, 4, 256), dtype=np.uint16)]
    ks, _, new_ctx = oracle.kv_commit(kc, kc, kn, kn, w.page_table, w.ctx_lens, w.q_indptr, [9],
                                      [list(range(9))])
    seq = oracle.gather_context(ks[0], w.page_table[0], int(new_ctx[0]))
    before = oracle.gather_context(kc[0], w.page_table[0], 29)
    np.testing.assert_array_equal(seq, np.concatenate([before, kn[0].astype(np.float64)]))


def test_commit_rejects_target_outside_pool():
    w = synth.make_structure(1, [14], [synth.chain_parents(1)], 3, 10, [0.9])
    bad = w.page_table.copy()
    bad[0, 0] = w.num_pool_pages
    c = [np.zeros((w.num_pool_pages, 4, 16, 256), np.uint16)]
    n = [np.zeros((2, 4, 256), np.uint16)]
    with pytest.raises(ValueError):
        oracle.kv_commit(c, c, n, n, bad, w.ctx_lens, w.q_indptr, [1], [[0]])
