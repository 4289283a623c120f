"""GPU sliding-window verify attention (through the C ABI) against the fp64 oracle.

Element by element on cases where the window cuts mid-tile and mid-page, is
narrower than the draft tree's depth, covers the whole context, or leaves a
split without any visible key for some columns; and sampled outputs at the
windowed workload's full size.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verify_decode_gb300 import synth

from gpu_helpers import check_attention, ensure_built, gpu_attention, oracle_attention, workload, f64, attn_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _tree(seed, budget):
    return synth.ddtree_parents(np.random.default_rng(seed), budget)[0]


CASES = {
    # name: (parents per sequence, ctx per sequence, window, forced splits)
    "chain8_ctx3000_w300": ([synth.chain_parents(8)], [3000], 300, 0),
    "chain8_ctx3000_w300_one_split": ([synth.chain_parents(8)], [3000], 300, 1),
    "tree22_ctx2500_w137_splits5": ([_tree(11, 22)], [2500], 137, 5),
    "tree22_ctx900_w3": ([_tree(12, 22)], [900], 3, 0),
    "tree63_ctx500_w20": ([_tree(13, 63)], [500], 20, 2),
    "chain4_ctx100_w1": ([synth.chain_parents(4)], [100], 1, 0),
    "wide_window_whole_context": ([_tree(14, 22)], [777], 5000, 0),
    "ragged_batch_w250": ([synth.chain_parents(0), synth.chain_parents(4), _tree(15, 22), synth.chain_parents(8)],
                          [0, 17, 1500, 4100], 250, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_window_attention_matches_oracle(name):
    parents, ctx, window, splits = CASES[name]
    w = workload(parents, ctx, seed=len(name) + 7, scale=1.0)
    out, lse, status = gpu_attention(w, 0, num_splits=splits, window=window)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0, window=window)
    check_attention(out, ref, lse, ref_lse)


def test_windowed_workload_full_size_sampled():
    w = synth.make_workload("chain8_ctx32k_win2048", device="cuda", layers=1, logits=False)
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    got = f64(out)
    assert np.isfinite(got).all()
    samples = [(r, h) for r in range(w.total_nodes) for h in (0, 7, 23)]
    ref, ref_lse = oracle_attention(w, 0, samples=samples)
    sub = np.stack([got[r, h] for r, h in samples])
    err = float(np.abs(sub - ref).max())
    assert err <= attn_bound(ref)
    assert err <= 1e-2 * float(np.abs(ref).max()) + 1e-6, err
