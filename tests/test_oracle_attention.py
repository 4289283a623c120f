"""Pins for the oracle's verify attention, independent of the oracle itself.

* closed forms: one visible key returns its value; q = 0 gives the plain mean
  of the visible values and lse = log(count); equal scores give the mean and
  lse = s + log(count) for a score fixed by construction;
* a chain draft block equals bottom-right-aligned causal attention from
  torch's scaled_dot_product_attention (fp64, KV heads repeated 6x), the case
  whose misalignment the 14->159 tok/s notes report as a FlashAttention-2
  off-by-one («Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图», 5.3);
* a tree equals SDPA under a mask built from the transitive closure of the
  parent relation (a construction independent of the oracle's parent walk);
* identity and permuted page tables give identical results (16-token pages
  from one pool, same page, sections 2 and 4).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_decode_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _f64(t):
    return t.to(torch.float64).numpy()


def _mk(parents_list, ctx, seed, scale=1.0, table="permuted", spare=0):
    w = synth.make_structure(len(parents_list), ctx, parents_list, seed, 64, [0.5] * len(parents_list),
                             table=table, spare_pages=spare)
    return synth.fill_tensors(w, 1, seed, qkv_scale=scale, logits=False)


def _run(w):
    return oracle.verify_attention(_f64(w.q[0]), _f64(w.k_cache[0]), _f64(w.v_cache[0]),
                                   _f64(w.k_new[0]), _f64(w.v_new[0]), w.page_table, w.ctx_lens,
                                   w.q_indptr, w.parents)


def _contiguous_context(w, b, layer_cache):
    """The context of sequence b as [L, 4, D], read page by page in logical order."""
    L = int(w.ctx_lens[b])
    out = []
    for p in range(0, L, 16):
        page = int(w.page_table[b, p // 16])
        n = min(16, L - p)
        out.append(_f64(layer_cache[page, :, :n, :]).transpose(1, 0, 2))
    return np.concatenate(out) if out else np.zeros((0, 4, 256))


def _closure(parents):
    """anc[j, i] = 1 iff i is j or an ancestor of j (boolean matrix powers)."""
    n = len(parents)
    a = np.eye(n, dtype=bool)
    for j in range(1, n):
        a[j, parents[j]] = True
    for _ in range(n):
        a = (a.astype(np.int64) @ a.astype(np.int64)) > 0
    return a


def _sdpa(w, b, mask_draft):
    """Reference attention of sequence b from torch SDPA with an explicit mask."""
    lo, hi = int(w.q_indptr[b]), int(w.q_indptr[b + 1])
    n = hi - lo
    L = int(w.ctx_lens[b])
    kc = _contiguous_context(w, b, w.k_cache[0])
    vc = _contiguous_context(w, b, w.v_cache[0])
    k = np.concatenate([kc, _f64(w.k_new[0])[lo:hi]])       # [L+n, 4, D]
    v = np.concatenate([vc, _f64(w.v_new[0])[lo:hi]])
    q = torch.from_numpy(_f64(w.q[0])[lo:hi]).permute(1, 0, 2)  # [24, n, D]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(6, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(6, dim=0)
    mask = torch.ones((n, L + n), dtype=torch.bool)
    mask[:, L:] = torch.from_numpy(mask_draft)
    out = torch.nn.functional.scaled_dot_product_attention(q, kt, vt, attn_mask=mask)
    return out.permute(1, 0, 2).numpy()


def test_single_visible_key_returns_its_value():
    w = _mk([np.array([-1], dtype=np.int32)], [0], seed=11, scale=1.0)
    o, lse = _run(w)
    for h in range(24):
        np.testing.assert_array_equal(o[0, h], _f64(w.v_new[0])[0, h // 6])


def test_zero_query_gives_mean_of_visible_values_and_log_count():
    par = synth.ddtree_parents(np.random.default_rng(3), 12)[0]
    w = _mk([par], [37], seed=12, scale=1.0)
    w.q[0].zero_()
    o, lse = _run(w)
    anc = _closure(par)
    kc = _contiguous_context(w, 0, w.v_cache[0])
    for j in range(len(par)):
        vis = np.concatenate([kc, _f64(w.v_new[0])[np.flatnonzero(anc[j])]])
        for h in range(24):
            np.testing.assert_allclose(o[j, h], vis[:, h // 6].mean(axis=0), rtol=0, atol=1e-15)
            assert lse[j, h] == pytest.approx(math.log(37 + anc[j].sum()), abs=1e-13)


def test_equal_scores_give_mean_and_shifted_log_count():
    # q = a e_0 and every key = c e_0 (+ noise off axis 0 that q does not see):
    # every score is a*c/16, so o is the plain mean and lse = a*c/16 + log(n).
    par = synth.chain_parents(3)
    w = _mk([par], [21], seed=13, scale=1.0)
    a, c = 3.0, 2.5
    w.q[0].zero_()
    w.q[0][..., 0] = a
    for t in (w.k_cache[0], w.k_new[0]):
        t[..., 0] = c
        t[..., 1:] = 0
    o, lse = _run(w)
    vc = _contiguous_context(w, 0, w.v_cache[0])
    for j in range(4):
        vis = np.concatenate([vc, _f64(w.v_new[0])[: j + 1]])
        for h in (0, 5, 6, 23):
            np.testing.assert_allclose(o[j, h], vis[:, h // 6].mean(axis=0), atol=1e-15)
            assert lse[j, h] == pytest.approx(a * c / 16 + math.log(21 + j + 1), abs=1e-13)


@pytest.mark.parametrize("ctx,k", [(0, 4), (5, 4), (53, 8), (100, 1)])
def test_chain_equals_bottom_right_causal_sdpa(ctx, k):
    par = synth.chain_parents(k)
    w = _mk([par], [ctx], seed=20 + ctx, scale=1.0)
    o, _ = _run(w)
    n = k + 1
    causal = torch.ones((n, n), dtype=torch.bool).tril().numpy()
    ref = _sdpa(w, 0, causal)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_equals_sdpa_with_closure_mask(seed):
    rng = np.random.default_rng(seed)
    par = synth.ddtree_parents(rng, 22)[0]
    par2 = synth.chain_parents(2)
    w = _mk([par, par2], [45, 19], seed=30 + seed, scale=0.7)
    o, _ = _run(w)
    np.testing.assert_allclose(o[:23], _sdpa(w, 0, _closure(par)), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o[23:], _sdpa(w, 1, _closure(par2)), rtol=1e-12, atol=1e-13)


def test_page_permutation_invariance():
    par = synth.chain_parents(4)
    wi = _mk([par, par], [70, 33], seed=40, table="identity", spare=3)
    wp = _mk([par, par], [70, 33], seed=40, table="identity", spare=3)
    # move every page of wp to a random physical page, keeping contents
    perm = np.random.default_rng(5).permutation(wp.num_pool_pages)
    for c in (wp.k_cache, wp.v_cache):
        moved = torch.empty_like(c[0])
        moved[torch.from_numpy(perm)] = c[0]
        c[0] = moved
    wp.page_table = np.where(wp.page_table >= 0, perm[np.maximum(wp.page_table, 0)], -1).astype(np.int32)
    oi, li = _run(wi)
    op, lp = _run(wp)
    np.testing.assert_array_equal(oi, op)
    np.testing.assert_array_equal(li, lp)


def test_samples_match_full_result():
    par = synth.ddtree_parents(np.random.default_rng(9), 10)[0]
    w = _mk([synth.chain_parents(4), par], [40, 17], seed=50, scale=1.0)
    o, lse = _run(w)
    samples = [(0, 0), (3, 7), (5, 23), (15, 12)]
    os_, ls = oracle.verify_attention(_f64(w.q[0]), _f64(w.k_cache[0]), _f64(w.v_cache[0]),
                                      _f64(w.k_new[0]), _f64(w.v_new[0]), w.page_table, w.ctx_lens,
                                      w.q_indptr, w.parents, samples=samples)
    for i, (r, h) in enumerate(samples):
        np.testing.assert_array_equal(os_[i], o[r, h])
        assert ls[i] == lse[r, h]


def test_invalid_parents_rejected():
    for bad in ([0, 0], [-1, 1], [-1, 0, 3], [-1, -1]):
        with pytest.raises(ValueError):
            oracle.tree_ancestors(np.array(bad))
