"""Oracle for the tree-aware Gated DeltaNet verify of the hybrid model's linear-attention layers.

TEST INFRASTRUCTURE ONLY.  Plain, slow CPU reference in float64; only the tests, the smoke check and the
bench's CPU-baseline leg may import it.  It shares no code with the CUDA path and imports nothing from the
product package.

Source: «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (S5).  [为什么我们要做这个测试]: 48 of
the model's 64 layers are Gated DeltaNet layers, which keep a recurrent (SSM) state cache besides the KV
cache.  [关键突破]: the verify step runs them over the draft tree with a tree-aware kernel that writes the
accepted state in place ("persist"), and a tree-aware short convolution in which each node gathers its
convolution window along its own parent chain instead of in DFS order.

The page names these kernels but gives no formulas.  Readings (each is also listed in the design notes):

* the recurrence is the published Gated DeltaNet rule, per value head, with state S (d_v x d_k):
      S_t = alpha_t * S_{t-1} + beta_t * (v_t - alpha_t * S_{t-1} k_t) k_t^T,   o_t = S_t q_t,
  alpha_t = exp(g_t) with g_t <= 0 given, beta_t in [0, 1] given, q and k L2-normalised per head (a zero
  vector stays zero) and q scaled by 1 / sqrt(d_k);
* on a tree, S_{t-1} is the state of the node's parent; the root's parent state is the cached state;
* value head h reads key head h // (H_v / H_k);
* the short convolution is causal and depthwise with 4 taps followed by SiLU:
      y_t[c] = silu(sum_i w[c][i] * x_{t-3+i}[c]),
  where, on a tree, x_{t-1}, x_{t-2}, x_{t-3} are the inputs of the node's parent, grandparent, ..., and
  past the root the cached convolution state (the last three committed inputs, oldest first);
* persist-on-accept: after the step accepts path p_0 .. p_{A-1}, the recurrent state becomes the state of
  node p_{A-1} and the convolution state the last three inputs of (old state, x_{p_0}, .., x_{p_{A-1}}).
"""
from __future__ import annotations

import math

import numpy as np


def l2norm(x):
    """x / ||x|| along the last axis; a zero vector stays zero."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)


def gdn_tree(q, k, v, g, beta, state, q_indptr, parents):
    """Gated DeltaNet over each sequence's draft tree.

    q, k: [sumN, H_k, d_k]; v: [sumN, H_v, d_v]; g, beta: [sumN, H_v]; state: [B, H_v, d_v, d_k];
    parents: [sumN] local ids (root -1).  Returns (o [sumN, H_v, d_v], states [sumN, H_v, d_v, d_k]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    state = np.asarray(state, dtype=np.float64)
    n_total, hk, dk = q.shape
    hv = v.shape[1]
    group = hv // hk
    o = np.zeros((n_total, hv, v.shape[2]))
    states = np.zeros((n_total, hv, v.shape[2], dk))
    for b in range(len(q_indptr) - 1):
        lo, hi = int(q_indptr[b]), int(q_indptr[b + 1])
        for j in range(lo, hi):
            p = int(parents[j])
            for h in range(hv):
                s_prev = state[b, h] if p < 0 else states[lo + p, h]
                kh = l2norm(k[j, h // group])
                qh = l2norm(q[j, h // group]) / math.sqrt(dk)
                a = math.exp(g[j, h])
                s = a * s_prev + beta[j, h] * np.outer(v[j, h] - a * (s_prev @ kh), kh)
                states[j, h] = s
                o[j, h] = s @ qh
    return o, states


def gdn_commit(state, states, q_indptr, accept_len, paths):
    """New recurrent state per sequence: the state of its last accepted node."""
    out = np.array(state, dtype=np.float64, copy=True)
    for b in range(len(q_indptr) - 1):
        last = paths[b][int(accept_len[b]) - 1]
        out[b] = states[int(q_indptr[b]) + last]
    return out


def silu(x):
    return x / (1.0 + np.exp(-x))


def conv_tree(x, w, conv_state, q_indptr, parents):
    """Causal 4-tap depthwise convolution + SiLU along each node's parent chain.

    x: [sumN, C]; w: [C, 4] (w[:, 3] multiplies the node's own input); conv_state: [B, C, 3] (oldest
    first).  Returns y [sumN, C].
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    conv_state = np.asarray(conv_state, dtype=np.float64)
    y = np.zeros_like(x)
    for b in range(len(q_indptr) - 1):
        lo, hi = int(q_indptr[b]), int(q_indptr[b + 1])
        for j in range(lo, hi):
            window = []                       # newest first: x_t, x_{t-1}, x_{t-2}, x_{t-3}
            u = j - lo
            while len(window) < 4 and u >= 0:
                window.append(x[lo + u])
                u = int(parents[lo + u])
            back = 2
            while len(window) < 4:
                window.append(conv_state[b, :, back])
                back -= 1
            acc = sum(w[:, 3 - i] * window[i] for i in range(4))
            y[j] = silu(acc)
    return y


def conv_commit(conv_state, x, q_indptr, accept_len, paths):
    """New convolution state: the last three inputs of (old state, accepted nodes' inputs)."""
    conv_state = np.asarray(conv_state)
    out = np.array(conv_state, copy=True)
    for b in range(len(q_indptr) - 1):
        seq = [conv_state[b, :, i] for i in range(3)]
        seq += [np.asarray(x)[int(q_indptr[b]) + paths[b][i]] for i in range(int(accept_len[b]))]
        for i in range(3):
            out[b, :, i] = seq[len(seq) - 3 + i]
    return out
