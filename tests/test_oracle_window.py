"""Pins of the oracle's sliding-window verify attention (CPU, not GPU).

The reading: node j sits at position L + depth(j); with window W it sees the
keys at its W most recent positions, its own included («如何在单张 RTX 3090 上让
Qwen3.5-27B token 生成速度提升 6 倍», 补充测试: attention over the most recent
2,048 KV positions).  Pinned by: a window wider than every position equals full
attention; W = 1 leaves each node its own key (o = its v); the root's output
equals full attention over a cache holding only the last W - 1 context tokens;
a chain equals SDPA under the banded causal mask; a tree equals SDPA under the
ancestor closure cut to the band.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_decode_gb300 import synth

from test_oracle_attention import _closure, _contiguous_context, _f64, _mk


def _run(w, window=None):
    return oracle.verify_attention(_f64(w.q[0]), _f64(w.k_cache[0]), _f64(w.v_cache[0]),
                                   _f64(w.k_new[0]), _f64(w.v_new[0]), w.page_table, w.ctx_lens,
                                   w.q_indptr, w.parents, window=window)


def _depths(par):
    d = np.zeros(len(par), dtype=np.int64)
    for j in range(1, len(par)):
        d[j] = d[par[j]] + 1
    return d


def _sdpa_band(w, b, par, window):
    """SDPA of sequence b with the mask: closure of the tree, cut to the window band."""
    lo, hi = int(w.q_indptr[b]), int(w.q_indptr[b + 1])
    n = hi - lo
    L = int(w.ctx_lens[b])
    k = np.concatenate([_contiguous_context(w, b, w.k_cache[0]), _f64(w.k_new[0])[lo:hi]])
    v = np.concatenate([_contiguous_context(w, b, w.v_cache[0]), _f64(w.v_new[0])[lo:hi]])
    depth = _depths(par)
    key_pos = np.concatenate([np.arange(L), L + depth])
    q_pos = L + depth
    band = (key_pos[None, :] <= q_pos[:, None]) & (key_pos[None, :] > q_pos[:, None] - window)
    allowed = np.ones((n, L + n), dtype=bool)
    allowed[:, L:] = _closure(par)
    mask = torch.from_numpy(band & allowed)
    q = torch.from_numpy(_f64(w.q[0])[lo:hi]).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(6, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(6, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(q, kt, vt, attn_mask=mask)
    return out.permute(1, 0, 2).numpy()


def test_wide_window_equals_full_attention():
    par = synth.ddtree_parents(np.random.default_rng(3), 12)[0]
    w = _mk([par, synth.chain_parents(4)], [77, 40], seed=50)
    full_o, full_lse = _run(w)
    o, lse = _run(w, window=77 + 16 + 1)
    np.testing.assert_array_equal(o, full_o)
    np.testing.assert_array_equal(lse, full_lse)


def test_window_one_keeps_only_the_own_key():
    par = synth.ddtree_parents(np.random.default_rng(4), 9)[0]
    w = _mk([par], [33], seed=51)
    o, lse = _run(w, window=1)
    k_new, v_new, q = _f64(w.k_new[0]), _f64(w.v_new[0]), _f64(w.q[0])
    for j in range(len(par)):
        for h in range(24):
            np.testing.assert_array_equal(o[j, h], v_new[j, h // 6])
            assert lse[j, h] == pytest.approx(float(q[j, h] @ k_new[j, h // 6]) / 16, abs=1e-12)


@pytest.mark.parametrize("L,window", [(100, 37), (64, 16), (200, 100)])
def test_root_equals_full_attention_over_the_last_tokens(L, window):
    """The root (position L) with window W sees context L-W+1..L-1 and itself:
    full attention over a second cache that holds only those W - 1 tokens."""
    par = synth.chain_parents(3)
    w = _mk([par], [L], seed=52 + L)
    o, lse = _run(w, window=window)
    keep = window - 1
    t = _mk([par], [keep], seed=52 + L)          # same draft block, fresh cache of `keep` tokens
    # copy the last `keep` context tokens of w into t's pages, in order
    kc = _contiguous_context(w, 0, w.k_cache[0])[L - keep:]
    vc = _contiguous_context(w, 0, w.v_cache[0])[L - keep:]
    for p in range(keep):
        page, slot = int(t.page_table[0, p // 16]), p % 16
        t.k_cache[0][page, :, slot, :] = torch.from_numpy(kc[p]).to(t.k_cache[0].dtype)
        t.v_cache[0][page, :, slot, :] = torch.from_numpy(vc[p]).to(t.v_cache[0].dtype)
    for attr in ("q", "k_new", "v_new"):
        getattr(t, attr)[0].copy_(getattr(w, attr)[0])
    ref_o, ref_lse = _run(t)
    np.testing.assert_allclose(o[0], ref_o[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse[0], ref_lse[0], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("L,k,window", [(90, 8, 20), (40, 4, 3), (130, 8, 129)])
def test_chain_equals_banded_causal_sdpa(L, k, window):
    par = synth.chain_parents(k)
    w = _mk([par], [L], seed=60 + window)
    o, _ = _run(w, window=window)
    np.testing.assert_allclose(o, _sdpa_band(w, 0, par, window), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("seed,window", [(0, 5), (1, 50), (2, 2)])
def test_tree_equals_sdpa_with_band_cut_closure(seed, window):
    par = synth.ddtree_parents(np.random.default_rng(seed), 22)[0]
    w = _mk([par], [70], seed=70 + seed, scale=0.7)
    o, _ = _run(w, window=window)
    np.testing.assert_allclose(o, _sdpa_band(w, 0, par, window), rtol=1e-12, atol=1e-13)
