"""Pins of the draft-tree construction oracle (CPU).

Top-K equals a stable numpy sort; log-sum-exp equals scipy's; with K = 1 the
tree is the greedy chain (the page's budget-15, K = 1 fast path); on small
inputs the tree's nodes equal a brute-force choice: every prefix of ranks
scored by its summed log-probabilities, the chain first, then the best
remaining prefixes; scores never rise along a root path; the tree is
prefix-closed with parent[j] < j.
"""
import itertools

import numpy as np
import pytest

import oracle.ddtree_oracle as dd


def _logits(rng, positions, vocab, scale=2.0):
    return rng.normal(0.0, scale, size=(positions, vocab))


def test_topk_matches_stable_sort_and_breaks_ties_by_index():
    rng = np.random.default_rng(0)
    x = rng.normal(size=1000)
    np.testing.assert_array_equal(dd.topk_first(x, 8), np.argsort(-x, kind="stable")[:8])
    y = np.array([1.0, 3.0, 3.0, 2.0, 3.0, -1.0])
    np.testing.assert_array_equal(dd.topk_first(y, 4), [1, 2, 4, 3])
    with pytest.raises(ValueError):
        dd.topk_first(np.array([0.0, np.nan]), 1)


def test_logsumexp_matches_scipy():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(1)
    x = rng.normal(0, 5, size=151936)
    assert dd.logsumexp(x) == pytest.approx(float(scipy_special.logsumexp(x)), rel=1e-13)


def test_k1_is_the_greedy_chain():
    rng = np.random.default_rng(2)
    logits = _logits(rng, 16, 500)
    par, tok, _, _ = dd.ddtree(logits, 1, 15, root_token=7)
    np.testing.assert_array_equal(par, np.arange(-1, 15))
    np.testing.assert_array_equal(tok, [7] + list(np.argmax(logits, axis=1)[:15]))


def _brute_force_ranks(cand_lp, budget):
    """All rank sequences (r_1..r_d), d <= positions; the chain (0,...,0) up to min(P, budget), then
    the best remaining ones by summed log-probability."""
    positions, k = cand_lp.shape
    prefixes = []
    for d in range(1, positions + 1):
        for ranks in itertools.product(range(k), repeat=d):
            prefixes.append((sum(cand_lp[i, r] for i, r in enumerate(ranks)), ranks))
    chain = [tuple([0] * d) for d in range(1, min(positions, budget) + 1)]
    rest = sorted((p for p in prefixes if p[1] not in set(chain)), key=lambda p: -p[0])
    return set(chain) | {r for _, r in rest[:budget - len(chain)]}


def _node_ranks(par, tok, cand_tok):
    """Rank sequence of every non-root node, recovered from parents and tokens."""
    out = []
    ranks = {0: ()}
    for j in range(1, len(par)):
        d = len(ranks[par[j]])
        r = int(np.flatnonzero(cand_tok[d] == tok[j])[0])
        ranks[j] = ranks[par[j]] + (r,)
        out.append(ranks[j])
    return out


@pytest.mark.parametrize("positions,k,budget,seed", [(3, 3, 8, 3), (4, 2, 9, 4), (4, 3, 14, 5), (2, 3, 11, 6),
                                                       (5, 2, 4, 7)])
def test_tree_equals_brute_force_prefix_choice(positions, k, budget, seed):
    rng = np.random.default_rng(seed)
    logits = _logits(rng, positions, 40)
    ct, cl = dd.candidates(logits, k)
    par, tok, sc, _ = dd.build_tree(ct, cl, budget, root_token=0)
    total = sum(k ** d for d in range(1, positions + 1))
    assert len(par) == 1 + min(budget, total)
    got = _node_ranks(par, tok, ct)
    assert len(set(got)) == len(got)
    assert set(got) == _brute_force_ranks(cl, budget)


@pytest.mark.parametrize("seed", [8, 9, 10])
def test_tree_invariants_at_the_page_sizes(seed):
    """16 positions, K = 8, budget 22 (the page's DDTree shape): parent[j] < j, scores never rise
    along a path and equal the summed log-probabilities, the chain is present, tokens match ranks."""
    rng = np.random.default_rng(seed)
    logits = _logits(rng, 16, 3000)
    ct, cl = dd.candidates(logits, 8)
    par, tok, sc, margin = dd.build_tree(ct, cl, 22, root_token=1)
    assert len(par) == 23 and par[0] == -1
    assert all(0 <= par[j] < j for j in range(1, 23))
    for j, ranks in enumerate(_node_ranks(par, tok, ct), start=1):
        assert sc[j] == pytest.approx(sum(cl[i, r] for i, r in enumerate(ranks)), abs=1e-12)
        assert sc[j] <= sc[par[j]] + 1e-15
    np.testing.assert_array_equal(tok[1:17], ct[:16, 0])          # the chain pre-seed
    np.testing.assert_array_equal(par[1:17], np.arange(0, 16))
    assert margin > 0
