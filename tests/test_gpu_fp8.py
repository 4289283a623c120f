"""Quantised (e4m3) KV cache on the GPU, through the C ABI, against the oracle.

Quantise-on-commit is compared byte for byte (round to nearest even,
saturation, signed zero, exact ties); the verify attention over e4m3 caches
element by element on cases that span several tiles and splits with ragged
tails, on a cache holding every finite code (subnormals, -0, +-448), and on
sampled outputs at the full sizes of the quantised workloads in the bench's
launch configuration.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_oracle as f8
from speculative_decoding_verify_decode_gb300 import native, synth
from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs

from gpu_helpers import (LSE_TOL, attn_bound, check_attention, ensure_built, f32, f64, gpu_attention,
                         oracle_attention, workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _tree(seed, budget):
    return synth.ddtree_parents(np.random.default_rng(seed), budget)[0]


# ---------------------------------------------------------------- commit

def _commit_case(parents_list, ctx, seed, k_scales, v_scales, special=None):
    """Run sd_kv_commit_fp8 on a planted accept result; returns (codes before, after, inputs)."""
    w = workload(parents_list, ctx, seed=seed, layers=len(k_scales), kv="fp8", logits=True)
    w.k_scales, w.v_scales = list(k_scales), list(v_scales)
    if special is not None:
        special(w)
    d = device_inputs(w)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, w.layers, w.vocab, k_scales=w.k_scales,
                    v_scales=w.v_scales)
    st.accept(w.logits, d["parents"], d["draft_tokens"])
    kc0 = [t.clone() for t in w.k_cache]
    vc0 = [t.clone() for t in w.v_cache]
    st.commit(w.k_cache, w.v_cache, w.k_new, w.v_new, d["page_table"], d["ctx_lens"])
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    _, lens, paths, _ = oracle.accept(w.q_indptr, w.parents, w.draft_tokens, w.logits.cpu().numpy())
    assert list(st.accept_len.cpu().numpy()) == list(lens)
    u8 = lambda ts: [t.cpu().numpy() for t in ts]
    ref_k, ref_v, ref_ctx = f8.kv_commit_fp8(u8(kc0), u8(vc0), w.k_scales, w.v_scales,
                                             [f32(t) for t in w.k_new], [f32(t) for t in w.v_new], w.page_table,
                                             w.ctx_lens, w.q_indptr, lens, paths)
    assert list(st.new_ctx_lens.cpu().numpy()) == list(ref_ctx)
    return u8(w.k_cache), u8(w.v_cache), ref_k, ref_v


def test_commit_bytes_match_the_oracle():
    got_k, got_v, ref_k, ref_v = _commit_case([synth.chain_parents(8), _tree(1, 22), synth.chain_parents(0)],
                                              [37, 511, 0], seed=3, k_scales=[0.0173, 2.0 ** -7],
                                              v_scales=[0.021, 0.0009])
    for a, b in zip(got_k + got_v, ref_k + ref_v):
        np.testing.assert_array_equal(a, b)


def test_commit_ties_saturation_and_zero_signs():
    """Power-of-two scales make x * (1 / scale) exact, so the planted rows hit exact
    e4m3 midpoints (ties to the even code), values beyond 448, infinities and -0."""
    mids = []
    for c in range(0x00, 0x7E):
        lo, hi = f8.e4m3_decode(c), f8.e4m3_decode(c + 1)
        mids += [(lo + hi) / 2, -(lo + hi) / 2]
    extra = [448.0, 456.0, 464.0, 480.0, 8192.0, -8192.0, float("inf"), float("-inf"), 0.0, -0.0, 2.0 ** -10,
             -(2.0 ** -10), 3 * 2.0 ** -11]
    vals = np.array(mids + extra, dtype=np.float64)
    scale = 2.0 ** -5

    def plant(w):
        for t in w.k_new + w.v_new:
            flat = t.view(-1)
            row = torch.tensor((vals * scale).astype(np.float32)).to(torch.bfloat16)
            assert np.array_equal(row.float().numpy().astype(np.float64), (vals * scale).astype(np.float32)), \
                "every planted value is exact in bf16"
            flat[: row.numel()] = row.to(flat.device)
            flat[2048: 2048 + row.numel()] = row.flip(0).to(flat.device)

    got_k, got_v, ref_k, ref_v = _commit_case([synth.chain_parents(8)], [21], seed=4, k_scales=[scale],
                                              v_scales=[scale], special=plant)
    for a, b in zip(got_k + got_v, ref_k + ref_v):
        np.testing.assert_array_equal(a, b)
    codes = set(np.unique(ref_k[0]).tolist())
    assert 0x7E in codes and 0xFE in codes and 0x80 in codes   # saturation both ways, and -0 kept


def test_commit_nan_gives_a_nan_code():
    def plant(w):
        for t in w.k_new:
            t.view(-1)[:64] = float("nan")

    got_k, _, ref_k, _ = _commit_case([synth.chain_parents(4)], [5], seed=5, k_scales=[0.01], v_scales=[0.01],
                                      special=plant)
    nan_ref = (ref_k[0] & 0x7F) == 0x7F
    assert nan_ref.any()
    assert np.array_equal((got_k[0] & 0x7F) == 0x7F, nan_ref)      # NaN where the oracle has NaN (any sign)
    np.testing.assert_array_equal(got_k[0][~nan_ref], ref_k[0][~nan_ref])


# ---------------------------------------------------------------- attention

CASES = {
    # name: (parents per sequence, ctx per sequence, qkv scale, forced splits)
    "chain4_ctx512_auto": ([synth.chain_parents(4)], [512], 1 / 16, 0),
    "chain8_ctx1000_three_splits": ([synth.chain_parents(8)], [1000], 1.0, 3),
    "tree22_ctx3000_five_splits": ([_tree(1, 22)], [3000], 1.0, 5),
    "ragged_batch_mixed_trees": ([synth.chain_parents(0), synth.chain_parents(4), _tree(3, 22),
                                  synth.chain_parents(8), _tree(4, 63)], [0, 1, 17, 700, 2049], 1.0, 0),
    "max_nodes64_ctx300": ([_tree(5, 63)], [300], 1.0, 2),
    "empty_context_tree": ([_tree(6, 22)], [0], 1.0, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_attention_matches_oracle(name):
    parents, ctx, scale, splits = CASES[name]
    w = workload(parents, ctx, seed=len(name), scale=scale, kv="fp8")
    if scale == 1.0:   # cache values near 1 as well, so that scores of order 1 make the softmax peaked
        w.k_scales = [16 * x for x in w.k_scales]
    out, lse, status = gpu_attention(w, 0, num_splits=splits)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0)
    check_attention(out, ref, lse, ref_lse)


def test_every_finite_code_is_read_back():
    """K and V hold every finite code (subnormals, -0, +-448), cycled through the pages."""
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    w = workload([_tree(8, 22), synth.chain_parents(8)], [700, 333], seed=8, kv="fp8")
    for i, t in enumerate(w.k_cache + w.v_cache):
        n = t.numel()
        pattern = np.resize(np.roll(finite, 37 * i), n)
        t.copy_(torch.from_numpy(pattern.reshape(t.shape)).to(t.device))
    w.k_scales, w.v_scales = [2.0 ** -9], [2.0 ** -8]    # keeps the +-448 keys' scores moderate
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0)
    check_attention(out, ref, lse, ref_lse)


@pytest.mark.parametrize("splits", [1, 4, 0])
def test_split_count_invariance(splits):
    w = workload([_tree(7, 22)], [2500], seed=77, scale=1.0, kv="fp8")
    base, base_lse, _ = gpu_attention(w, 0, num_splits=1)
    out, lse, status = gpu_attention(w, 0, num_splits=splits)
    assert status == 0
    ref = f64(base)
    assert float(np.abs(f64(out) - ref).max()) <= 1e-2 * float(np.abs(ref).max()) + 1e-6
    assert float(np.abs(f64(lse) - f64(base_lse)).max()) <= LSE_TOL


FULL = ["chain8_ctx4k_fp8", "ddtree22_ctx32k_fp8", "ddtree22_ctx128k_fp8"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full-size quantised workloads, bench launch configuration, sampled outputs vs the oracle."""
    w = synth.make_workload(name, device="cuda", layers=1, logits=False)
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    got = f64(out)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(6)
    n = w.total_nodes
    rows = sorted(set([0, n - 1] + list(rng.integers(0, n, size=8))))
    samples = [(int(r), int(h)) for r in rows for h in (0, 7, 12, 23)]
    ref, ref_lse = oracle_attention(w, 0, samples=samples)
    sub = np.stack([got[r, h] for r, h in samples])
    err = float(np.abs(sub - ref).max())
    assert err <= attn_bound(ref)
    assert err <= 1e-2 * float(np.abs(ref).max()) + 1e-6, err
    sub_lse = np.array([f64(lse)[r, h] for r, h in samples])
    assert float(np.abs(sub_lse - ref_lse).max()) <= LSE_TOL


def test_window_with_fp8_cache():
    w = workload([synth.chain_parents(8), _tree(9, 22)], [3000, 1900], seed=9, kv="fp8")
    w.window = 700
    out, lse, status = gpu_attention(w, 0)
    assert status == 0
    ref, ref_lse = oracle_attention(w, 0)
    check_attention(out, ref, lse, ref_lse)
