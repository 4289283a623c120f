"""GPU verify attention (through the C ABI) against the fp64 oracle.

Element by element on small cases that still span several KV tiles and
splits with ragged tails; sampled (row, head) outputs at the five workloads'
full sizes in the launch configuration the bench uses; and the invariance
of the result under the number of splits.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verify_decode_gb300 import synth

from gpu_helpers import (LSE_TOL, check_attention, ensure_built, gpu_attention, oracle_attention, workload, f64,
                         attn_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _tree(seed, budget):
    return synth.ddtree_parents(np.random.default_rng(seed), budget)[0]


CASES = {
    # name: (parents per sequence, ctx per sequence, qkv scale, forced splits)
    "chain4_ctx512_auto": ([synth.chain_parents(4)], [512], 1 / 16, 0),
    "chain8_ctx1000_one_split": ([synth.chain_parents(8)], [1000], 1.0, 1),
    "chain8_ctx1000_three_splits": ([synth.chain_parents(8)], [1000], 1.0, 3),
    "tree22_ctx3000_five_splits": ([_tree(1, 22)], [3000], 1.0, 5),
    "tree22_ctx3000_auto_spiky": ([_tree(2, 22)], [3000], 3.0, 0),
    "ragged_batch_mixed_trees": ([synth.chain_parents(0), synth.chain_parents(4), _tree(3, 22),
                                  synth.chain_parents(8), _tree(4, 63)], [0, 1, 17, 700, 2049], 1.0, 0),
    "max_nodes64_ctx300": ([_tree(5, 63)], [300], 1.0, 2),
    "empty_context_tree": ([_tree(6, 22)], [0], 1.0, 0),
    "ctx_one_page_exact": ([synth.chain_parents(4), synth.chain_parents(4)], [16, 64], 0.5, 0),
    # a chain over 4000 tokens: one tile per split (the automatic plan) runs attn_tc_kernel on bf16 caches,
    # three tiles per split the ring kernel
    "chain8_ctx4000_one_tile_splits": ([synth.chain_parents(8)], [4000], 1.0, 0),
    "chain8_ctx4000_three_tile_splits": ([synth.chain_parents(8)], [4000], 1.0, 11),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_attention_matches_oracle(name):
    parents, ctx, scale, splits = CASES[name]
    w = workload(parents, ctx, seed=len(name), scale=scale)
    out, lse, status = gpu_attention(w, 0, num_splits=splits)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0)
    check_attention(out, ref, lse, ref_lse)


def test_tiny_chain_workload_full():
    w = synth.make_workload("tiny_chain_ctx512", device="cuda")
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0)
    check_attention(out, ref, lse, ref_lse)


@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_split_count_invariance(splits):
    w = workload([_tree(7, 22)], [2500], seed=77, scale=1.0)
    base, base_lse, _ = gpu_attention(w, 0, num_splits=1)
    out, lse, status = gpu_attention(w, 0, num_splits=splits)
    assert status == 0
    ref = f64(base)
    assert float(np.abs(f64(out) - ref).max()) <= 1e-2 * float(np.abs(ref).max()) + 1e-6
    assert float(np.abs(f64(lse) - f64(base_lse)).max()) <= LSE_TOL


FULL = ["chain8_ctx4k", "ddtree22_ctx32k", "conc8_chain4_ragged", "ddtree22_ctx128k"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full-size shapes, bench launch configuration, sampled outputs vs the oracle."""
    w = synth.make_workload(name, device="cuda", layers=1, logits=False)
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    got = f64(out)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(5)
    n = w.total_nodes
    rows = sorted(set([0, n - 1] + list(rng.integers(0, n, size=10))))
    samples = [(int(r), int(h)) for r in rows for h in (0, 5, 6, 13, 23)]
    ref, ref_lse = oracle_attention(w, 0, samples=samples)
    sub = np.stack([got[r, h] for r, h in samples])
    err = float(np.abs(sub - ref).max())
    assert err <= attn_bound(ref)
    assert err <= 1e-2 * float(np.abs(ref).max()) + 1e-6, err
    sub_lse = np.array([f64(lse)[r, h] for r, h in samples])
    assert float(np.abs(sub_lse - ref_lse).max()) <= LSE_TOL


CHAIN_CASES = {
    # name: (kv, window, capture in a CUDA graph)
    "bf16_eager": ("bf16", 0, False),
    "bf16_graph": ("bf16", 0, True),
    "bf16_window300": ("bf16", 300, False),
    "fp8_eager": ("fp8", 0, False),
}


@pytest.mark.parametrize("name", sorted(CHAIN_CASES))
def test_layer_chain_with_early_context_loads(name):
    """Four layers issued back to back as a model issues them, every layer after the first with the
    context-stable flag (its context tiles load before the previous layer's merge has finished).  Each
    layer's queries are the previous layer's output buffer, pre-filled with NaN, and one workspace serves
    every layer, so a query read before the previous merge ends, or partials overwritten while that merge
    reads them, shows up.  The batch is ragged: an empty context, contexts of one split, several splits.
    The oracle runs the same chain on its own bf16-rounded outputs."""
    import oracle
    import oracle.fp8_oracle as fp8_oracle
    from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs

    kv, window, graph = CHAIN_CASES[name]
    layers = 4
    parents = [synth.chain_parents(0), synth.chain_parents(8), _tree(7, 22), synth.chain_parents(5)]
    w = workload(parents, [0, 100, 2500, 5000], seed=11 + len(name), scale=1.0, layers=layers, kv=kv)
    d = device_inputs(w)
    fp8 = kv == "fp8"
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, layers, max(w.vocab, 1), window=window,
                    k_scales=w.k_scales if fp8 else None, v_scales=w.v_scales if fp8 else None)

    def chain():
        for o in st.out:
            o.fill_(float("nan"))
        for layer in range(layers):
            q = w.q[0] if layer == 0 else st.out[layer - 1]
            st.attention(layer, q, w.k_cache[layer], w.v_cache[layer], w.k_new[layer], w.v_new[layer],
                         d["page_table"], d["ctx_lens"], d["parents"], ctx_stable=layer > 0)

    if graph:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            chain()   # warm-up outside the capture
            with torch.cuda.graph(g, stream=s):
                chain()
        torch.cuda.current_stream().wait_stream(s)
        run = g.replay
    else:
        run = chain

    q_ref = f64(w.q[0])
    refs = []
    for layer in range(layers):
        args = (w.k_new[layer], w.v_new[layer])
        if fp8:
            codes = lambda t: t.detach().cpu().numpy()
            ref, _ = fp8_oracle.verify_attention_fp8(q_ref, codes(w.k_cache[layer]), codes(w.v_cache[layer]),
                                                     w.k_scales[layer], w.v_scales[layer], f64(args[0]),
                                                     f64(args[1]), w.page_table, w.ctx_lens, w.q_indptr, w.parents,
                                                     window=window or None)
        else:
            ref, _ = oracle.verify_attention(q_ref, f64(w.k_cache[layer]), f64(w.v_cache[layer]), f64(args[0]),
                                             f64(args[1]), w.page_table, w.ctx_lens, w.q_indptr, w.parents,
                                             window=window or None)
        refs.append(ref)
        # the next layer's queries: this layer's output as the kernel stores it (bf16)
        q_ref = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()

    for _ in range(3):
        st.dev_status.zero_()
        run()
        torch.cuda.synchronize()
        assert int(st.dev_status.item()) == 0
        for layer in range(layers):
            got = f64(st.out[layer])
            assert np.isfinite(got).all(), layer
            err = float(np.abs(got - refs[layer]).max())
            # later layers also carry the previous layers' output rounding in their queries
            assert err <= attn_bound(refs[layer]), (layer, err, attn_bound(refs[layer]))
