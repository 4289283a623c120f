"""Pins of the tree Gated DeltaNet / tree convolution oracle (CPU).

Closed forms of the recurrence (no write: pure decay; unit write: the delta rule stores v exactly under
its key; orthonormal keys: an associative memory), an independent formulation of the same states (the
triangular system the chunked form solves, with decay ratios), tree = each node's root path run as a
chain, and for the convolution single-tap kernels, numpy's convolution on a chain and the commit's
last-three-inputs rule.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle.gdn_oracle as gd
from speculative_decoding_verify_decode_gb300 import synth


def _case(rng, parents_list, hk=2, hv=4, d=16, beta=None, g=None, zero_state=False):
    n = sum(len(p) for p in parents_list)
    indptr = np.concatenate([[0], np.cumsum([len(p) for p in parents_list])])
    parents = np.concatenate(parents_list)
    q = rng.normal(size=(n, hk, d))
    k = rng.normal(size=(n, hk, d))
    v = rng.normal(size=(n, hv, d))
    gg = -rng.uniform(0.0, 0.5, size=(n, hv)) if g is None else np.full((n, hv), g)
    bb = rng.uniform(0.0, 1.0, size=(n, hv)) if beta is None else np.full((n, hv), beta)
    state = np.zeros((len(parents_list), hv, d, d)) if zero_state else rng.normal(size=(len(parents_list), hv, d, d))
    return q, k, v, gg, bb, state, indptr, parents


def _tree(seed, budget):
    return synth.ddtree_parents(np.random.default_rng(seed), budget)[0]


def _path(parents, lo, j):
    out = []
    u = j - lo
    while u >= 0:
        out.append(u)
        u = int(parents[lo + u])
    return out[::-1]


def test_l2norm_and_silu():
    x = np.array([[3.0, 4.0], [0.0, 0.0]])
    np.testing.assert_allclose(gd.l2norm(x), [[0.6, 0.8], [0.0, 0.0]])
    z = np.linspace(-20, 20, 41)
    np.testing.assert_allclose(gd.silu(z), z * expit(z), rtol=1e-14, atol=1e-14)


def test_no_write_is_pure_decay():
    rng = np.random.default_rng(0)
    q, k, v, g, b, s0, ind, par = _case(rng, [_tree(1, 10), synth.chain_parents(5)], beta=0.0)
    o, _ = gd.gdn_tree(q, k, v, g, b, s0, ind, par)
    for s in range(2):
        lo, hi = ind[s], ind[s + 1]
        for j in range(lo, hi):
            path = _path(par, lo, j)
            for h in range(4):
                gamma = math.exp(sum(g[lo + m, h] for m in path))
                qh = q[j, h // 2] / np.linalg.norm(q[j, h // 2]) / 4.0
                np.testing.assert_allclose(o[j, h], gamma * s0[s, h] @ qh, rtol=1e-12, atol=1e-12)


def test_unit_write_stores_v_under_its_key():
    rng = np.random.default_rng(1)
    q, k, v, g, b, s0, ind, par = _case(rng, [_tree(2, 14)], beta=1.0)
    _, states = gd.gdn_tree(q, k, v, g, b, s0, ind, par)
    for j in range(len(par)):
        for h in range(4):
            kh = k[j, h // 2] / np.linalg.norm(k[j, h // 2])
            np.testing.assert_allclose(states[j, h] @ kh, v[j, h], rtol=1e-10, atol=1e-10)


def test_orthonormal_keys_are_an_associative_memory():
    rng = np.random.default_rng(2)
    d, n = 16, 6
    basis = np.linalg.qr(rng.normal(size=(d, d)))[0].T        # orthonormal rows
    par = synth.chain_parents(n - 1)
    q = np.zeros((n, 1, d)); k = np.zeros((n, 1, d)); v = rng.normal(size=(n, 1, d))
    for j in range(n):
        k[j, 0] = basis[j] * (1.0 + j)                        # any length: the key is normalised
        q[j, 0] = basis[(j * 3) % (j + 1)]                     # read an earlier (or the own) key
    o, _ = gd.gdn_tree(q, k, v, np.zeros((n, 1)), np.ones((n, 1)), np.zeros((1, 1, d, d)), [0, n], par)
    for j in range(n):
        np.testing.assert_allclose(o[j, 0], v[(j * 3) % (j + 1), 0] / 4.0, rtol=1e-12, atol=1e-12)


def test_matches_the_triangular_system_of_the_chunked_form():
    """u_j = beta_j (v_j - gamma_j S0 k_j - sum_{m < j on the path} (gamma_j / gamma_m)(k_m . k_j) u_m),
    o_j = gamma_j S0 q_j + sum_{m on the path, m <= j} (gamma_j / gamma_m)(k_m . q_j) u_m."""
    rng = np.random.default_rng(3)
    parents_list = [_tree(4, 22), synth.chain_parents(7), _tree(5, 30)]
    q, k, v, g, b, s0, ind, par = _case(rng, parents_list)
    o, _ = gd.gdn_tree(q, k, v, g, b, s0, ind, par)
    for s in range(len(parents_list)):
        lo, hi = ind[s], ind[s + 1]
        n = hi - lo
        for h in range(4):
            kh = np.stack([k[lo + j, h // 2] / np.linalg.norm(k[lo + j, h // 2]) for j in range(n)])
            qh = np.stack([q[lo + j, h // 2] / np.linalg.norm(q[lo + j, h // 2]) / 4.0 for j in range(n)])
            logg = np.zeros(n)
            anc = np.zeros((n, n), dtype=bool)                  # anc[j, m]: m on j's path, m < j
            for j in range(n):
                p = int(par[lo + j])
                logg[j] = g[lo + j, h] + (logg[p] if p >= 0 else 0.0)
                if p >= 0:
                    anc[j] = anc[p]
                    anc[j, p] = True
            ratio = np.exp(logg[:, None] - logg[None, :])
            L = np.where(anc, ratio * (kh @ kh.T), 0.0) * b[lo:hi, h][:, None]
            rhs = b[lo:hi, h][:, None] * (v[lo:hi, h] - np.exp(logg)[:, None] * (kh @ s0[s, h].T))
            U = np.linalg.solve(np.eye(n) + L, rhs)
            incl = anc | np.eye(n, dtype=bool)
            O = np.exp(logg)[:, None] * (qh @ s0[s, h].T) + np.where(incl, ratio * (qh @ kh.T), 0.0) @ U
            np.testing.assert_allclose(o[lo:hi, h], O, rtol=1e-9, atol=1e-9)


def test_tree_equals_each_root_path_run_as_a_chain():
    rng = np.random.default_rng(4)
    q, k, v, g, b, s0, ind, par = _case(rng, [_tree(6, 22)])
    o, _ = gd.gdn_tree(q, k, v, g, b, s0, ind, par)
    for j in range(len(par)):
        path = _path(par, 0, j)
        oc, _ = gd.gdn_tree(q[path], k[path], v[path], g[path], b[path], s0, [0, len(path)],
                            synth.chain_parents(len(path) - 1))
        np.testing.assert_allclose(o[j], oc[-1], rtol=1e-12, atol=1e-12)


def test_commit_takes_the_last_accepted_node():
    rng = np.random.default_rng(5)
    parents_list = [_tree(7, 12), synth.chain_parents(4)]
    q, k, v, g, b, s0, ind, par = _case(rng, parents_list)
    _, states = gd.gdn_tree(q, k, v, g, b, s0, ind, par)
    paths = [[0, 2, 5], [0, 1]]
    new = gd.gdn_commit(s0, states, ind, [3, 2], paths)
    np.testing.assert_array_equal(new[0], states[5])
    np.testing.assert_array_equal(new[1], states[ind[1] + 1])


def test_conv_single_taps_pick_the_right_inputs():
    rng = np.random.default_rng(6)
    par = _tree(8, 12)
    n, c = len(par), 5
    x = rng.normal(size=(n, c)); st = rng.normal(size=(1, c, 3))
    for tap in range(4):
        w = np.zeros((c, 4)); w[:, tap] = 1.0
        y = gd.conv_tree(x, w, st, [0, n], par)
        back = 3 - tap                                          # how many steps back this tap reads
        for j in range(n):
            path = _path(par, 0, j)
            src = x[path[-1 - back]] if back < len(path) else st[0, :, 3 - (back - len(path)) - 1]
            np.testing.assert_allclose(y[j], gd.silu(src), rtol=1e-14)


def test_conv_chain_matches_numpy_convolution():
    rng = np.random.default_rng(7)
    n, c = 9, 6
    x = rng.normal(size=(n, c)); w = rng.normal(size=(c, 4)); st = rng.normal(size=(1, c, 3))
    y = gd.conv_tree(x, w, st, [0, n], synth.chain_parents(n - 1))
    for ch in range(c):
        seq = np.concatenate([st[0, ch], x[:, ch]])
        full = np.convolve(seq, w[ch, ::-1], mode="valid")      # out_t = sum_i w[i] seq[t + i]
        np.testing.assert_allclose(y[:, ch], gd.silu(full), rtol=1e-12, atol=1e-12)


def test_conv_commit_keeps_the_last_three_inputs():
    rng = np.random.default_rng(8)
    c = 4
    x = rng.normal(size=(7, c)); st = rng.normal(size=(2, c, 3))
    new = gd.conv_commit(st, x, [0, 5, 7], [3, 1], [[0, 2, 4], [0]])
    np.testing.assert_array_equal(new[0], x[[0, 2, 4]].T)
    np.testing.assert_array_equal(new[1], np.stack([st[1, :, 1], st[1, :, 2], x[5]], axis=1))
