"""Pins of the sampling-verify oracle (CPU).

The rule must leave the target distribution unchanged: the first emitted token of a node whose children were
drawn from q is distributed as p — checked by Monte Carlo on a 5-token vocabulary for one child, for two
children (the multi-candidate rule) and for a chain.  Special cases: draft = target accepts every draft; a
draft token the target gives probability 0 is always rejected; a near-zero temperature with a draft that is
the greedy choice reduces to the greedy verify; inverse-CDF sampling on hand cases.
"""
import numpy as np
import pytest

import oracle
import oracle.sampling_oracle as so
from speculative_decoding_verify_decode_gb300 import synth


def _first_token_freq(p_logits, q, n_children, trials, seed, temperature=1.0):
    """Frequencies of the first emitted token when the root's children are drawn i.i.d. from q."""
    rng = np.random.default_rng(seed)
    V = len(q)
    counts = np.zeros(V)
    n = 1 + n_children
    parents = np.array([-1] + [0] * n_children)
    logits = np.zeros((n, V))
    logits[0] = p_logits
    dp = np.tile(q, (n, 1))
    dp[1:] = 1.0 / V        # the children's own draft rows (for grandchildren) must not enter the root's decisions
    for _ in range(trials):
        drafts = np.concatenate([[0], rng.choice(V, size=n_children, p=q)])
        # children are leaves: an accepted child emits its token, then samples a bonus at the child
        lens, paths, outs, _ = so.sampling_accept([0, n], parents, drafts, logits, dp, temperature,
                                                  rng.random(n), rng.random(n))
        counts[outs[0][0]] += 1
    return counts / trials


@pytest.mark.parametrize("n_children", [1, 2, 3])
def test_first_token_is_distributed_as_the_target(n_children):
    p_logits = np.log(np.array([0.05, 0.4, 0.1, 0.3, 0.15]))
    q = np.array([0.3, 0.1, 0.3, 0.1, 0.2])
    trials = 20000
    freq = _first_token_freq(p_logits, q, n_children, trials, seed=n_children)
    p = so.softmax_t(p_logits, 1.0)
    sigma = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(freq - p) <= 4.5 * sigma), (freq, p)


def test_chain_second_token_is_distributed_as_the_target():
    rng = np.random.default_rng(7)
    V, trials = 4, 20000
    l0 = np.log(np.array([0.5, 0.2, 0.2, 0.1]))
    l1 = np.log(np.array([0.1, 0.6, 0.2, 0.1]))
    q0 = np.array([0.25, 0.25, 0.25, 0.25])
    q1 = np.array([0.4, 0.2, 0.2, 0.2])
    counts = np.zeros(V)
    hits = 0
    for _ in range(trials):
        d1 = rng.choice(V, p=q0)
        d2 = rng.choice(V, p=q1)
        logits = np.stack([l0, l1, np.zeros(V)])
        lens, _, outs, _ = so.sampling_accept([0, 3], [-1, 0, 1], [0, d1, d2], logits, np.stack([q0, q1, q1]), 1.0,
                                              rng.random(3), rng.random(3))
        if outs[0][0] == 1:       # condition on the first token being 1: the second follows p(. | 1) = l1
            counts[outs[0][1]] += 1
            hits += 1
    p1 = so.softmax_t(l1, 1.0)
    sigma = np.sqrt(p1 * (1 - p1) / hits)
    assert np.all(np.abs(counts / hits - p1) <= 4.5 * sigma)


def test_draft_equal_to_target_accepts_everything():
    rng = np.random.default_rng(1)
    par = synth.ddtree_parents(rng, 12)[0]
    n, V = len(par), 50
    logits = rng.normal(size=(n, V))
    probs = np.stack([so.softmax_t(l, 0.7) for l in logits])
    # the deepest chain: every node's first child drafts a token with q = p at its parent
    drafts = rng.integers(0, V, size=n)
    lens, paths, _, _ = so.sampling_accept([0, n], par, drafts, logits, probs, 0.7, rng.random(n) * 0.999, rng.random(n))
    # the walk always takes the first child: the path is the first-child chain down to a leaf
    u, expect = 0, [0]
    while True:
        kids = [j for j in range(1, n) if par[j] == u]
        if not kids:
            break
        u = kids[0]
        expect.append(u)
    assert paths[0] == expect


def test_zero_probability_draft_is_rejected():
    V = 6
    logits = np.full((2, V), -np.inf)
    logits[:, :3] = 0.0                       # tokens 3.. have probability 0
    q = np.full((2, V), 1.0 / V)
    lens, _, outs, _ = so.sampling_accept([0, 2], [-1, 0], [0, 4], logits, q, 1.0, [0.0, 0.0], [0.5, 0.5])
    assert lens[0] == 1 and outs[0][0] in (0, 1, 2)


def test_near_zero_temperature_reduces_to_greedy():
    s = synth.make_structure(2, [16, 16], [synth.chain_parents(6), synth.ddtree_parents(np.random.default_rng(2), 10)[0]],
                             5, 300, [0.7, 0.7])
    V = 300
    rng = np.random.default_rng(3)
    n = s.total_nodes
    logits = rng.normal(size=(n, V))
    logits[np.arange(n), s.tau] += 4.0
    q = np.full((n, V), 1e-3 / (V - 1))
    for j in range(n):                         # the draft model puts its mass on the target's greedy choice
        q[j, s.tau[j]] = 1.0 - 1e-3
    tg, glens, gpaths, gtoks = oracle.accept(s.q_indptr, s.parents, s.draft_tokens, logits)
    lens, paths, outs, _ = so.sampling_accept(s.q_indptr, s.parents, s.draft_tokens, logits, q, 1e-3,
                                              np.full(n, 0.5), np.full(n, 0.5))
    assert list(lens) == list(glens)
    assert [list(x) for x in paths] == [list(x) for x in gpaths]
    assert [list(x) for x in outs] == [list(x) for x in gtoks]


def test_inverse_cdf_hand_cases():
    w = np.array([0.0, 1.0, 0.0, 3.0])
    assert so.inverse_cdf(w, 0.0) == 1
    assert so.inverse_cdf(w, 0.2499) == 1
    assert so.inverse_cdf(w, 0.25) == 3
    assert so.inverse_cdf(w, 0.999) == 3
