"""GPU parity at the workloads' stated shapes (through the C ABI), against the oracle.

* The long-context tree verify (131072 tokens of context, a 22-node tree) with
  its context cut into 64 chunks per KV head (256 split partials per layer,
  merged by their log-sum-exp weights), sampled outputs.
* The 32K tree workload with every (node row, query head) compared.
* Whole 16-layer verify steps at the 8-chain 4K and the 32K tree workloads'
  full shapes (full page pool, permuted page table): accept lengths, paths and
  emitted tokens bit for bit, and every byte of every layer's K and V cache
  after the commit.
* The error budget of bf16 split partials on a many-split case with spiky
  scores: a partial is rounded once to bf16 and the merged output once more,
  so the merge adds at most two bf16 roundings (2 x 2^-9 of the largest
  partial) to the single-split error.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_decode_gb300 import synth
from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs

from gpu_helpers import LSE_TOL, attn_bound, ensure_built, f64, gpu_attention, oracle_attention, tight_bound, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _compare(out, lse, ref, ref_lse, bound):
    got = f64(out)
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max())
    assert err <= attn_bound(ref), (err, attn_bound(ref))
    assert err <= bound, (err, bound)
    lerr = float(np.abs(f64(lse) - ref_lse).max())
    assert lerr <= LSE_TOL, lerr
    return err


def test_long_context_tree_with_64_chunks_per_kv_head():
    w = synth.make_workload("ddtree22_ctx128k", device="cuda", layers=1, logits=False)
    out, lse, status = gpu_attention(w, 0, num_splits=64)
    assert status == 0
    rng = np.random.default_rng(64)
    n = w.total_nodes
    rows = sorted(set([0, n - 1] + [int(x) for x in rng.integers(0, n, size=6)]))
    samples = [(r, h) for r in rows for h in range(0, 24, 5)]
    ref, ref_lse = oracle_attention(w, 0, samples=samples)
    got = f64(out)
    sub = np.stack([got[r, h] for r, h in samples])
    sub_lse = np.array([f64(lse)[r, h] for r, h in samples])
    err = float(np.abs(sub - ref).max())
    assert err <= attn_bound(ref) and err <= tight_bound(ref), err
    assert float(np.abs(sub_lse - ref_lse).max()) <= LSE_TOL


def test_tree_32k_every_row_and_head():
    w = synth.make_workload("ddtree22_ctx32k", device="cuda", layers=1, logits=False)
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0)
    _compare(out, lse, ref, ref_lse, tight_bound(ref))


def test_many_splits_bf16_partials_within_their_budget():
    """64 context chunks of a spiky-score tree: every chunk's partial output is rounded to bf16
    before the merge.  The merged output is a convex combination of the partials, so the two
    roundings add at most 2 * 2^-9 * max|partial|; the partials are bounded by the values, which
    are bounded by a few times max|ref| here.  The check: the many-split error stays within the
    single-split error plus 2^-7 * max|ref|."""
    w = workload([synth.ddtree_parents(np.random.default_rng(21), 22)[0]], [8192], seed=21, scale=3.0)
    ref, ref_lse = oracle_attention(w, 0)
    one, one_lse, st1 = gpu_attention(w, 0, num_splits=1)
    many, many_lse, st64 = gpu_attention(w, 0, num_splits=64)
    assert st1 == 0 and st64 == 0
    err1 = float(np.abs(f64(one) - ref).max())
    err64 = _compare(many, many_lse, ref, ref_lse, tight_bound(ref))
    assert err64 <= err1 + 2.0 ** -7 * float(np.abs(ref).max()), (err64, err1)


def _full_step(name):
    w = synth.make_workload(name, device="cuda")
    d = device_inputs(w)
    k0 = [t.view(torch.int16).cpu().numpy() for t in w.k_cache]
    v0 = [t.view(torch.int16).cpu().numpy() for t in w.v_cache]
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, w.layers, w.vocab)
    st.run(w.q, w.k_cache, w.v_cache, w.k_new, w.v_new, d["page_table"], d["ctx_lens"], d["parents"],
           d["draft_tokens"], w.logits)
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    t, lens, paths, toks = oracle.accept(w.q_indptr, w.parents, w.draft_tokens, w.logits.cpu().numpy())
    np.testing.assert_array_equal(st.target_tokens.cpu().numpy(), t)
    np.testing.assert_array_equal(st.accept_len.cpu().numpy(), lens)
    path, out_tok = st.path.cpu().numpy(), st.out_tokens.cpu().numpy()
    for b in range(w.batch):
        a = int(lens[b])
        assert list(path[b, :a]) == paths[b] and (path[b, a:] == -1).all()
        assert list(out_tok[b, :a]) == toks[b] and (out_tok[b, a:] == -1).all()
    new_ctx = None
    for layer in range(w.layers):   # one layer at a time keeps the host copies small
        kn = [w.k_new[layer].view(torch.int16).cpu().numpy()]
        vn = [w.v_new[layer].view(torch.int16).cpu().numpy()]
        ref_k, ref_v, new_ctx = oracle.kv_commit([k0[layer]], [v0[layer]], kn, vn, w.page_table, w.ctx_lens,
                                                 w.q_indptr, lens, paths)
        np.testing.assert_array_equal(w.k_cache[layer].view(torch.int16).cpu().numpy(), ref_k[0])
        np.testing.assert_array_equal(w.v_cache[layer].view(torch.int16).cpu().numpy(), ref_v[0])
        k0[layer] = v0[layer] = None
    np.testing.assert_array_equal(st.new_ctx_lens.cpu().numpy(), new_ctx)
    return lens


def test_full_step_chain8_4k_all_layers():
    lens = _full_step("chain8_ctx4k")
    assert 1 <= int(lens[0]) <= 9


def test_full_step_tree22_32k_all_layers():
    lens = _full_step("ddtree22_ctx32k")
    assert 1 <= int(lens[0]) <= 17
