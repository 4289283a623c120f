"""Sampling-based verify on the GPU, through the C ABI, against the oracle.

Decisions are compared exactly wherever the oracle's smallest decision margin (relative distance of an
acceptance test from its threshold, or distance of the bonus draw from a CDF boundary relative to the
total) exceeds 5e-5, above the fp32 rounding of the kernel's sums over the vocabulary (about 1e-5 at
152K tokens in the worst case); the rest must still be valid outputs.  Target rows put most of their
mass on three tokens over a flat tail.  Cases: chains and trees, a ragged batch with root-only sequences,
temperatures 0.5 to 2, the full vocabulary and sizes that are not a multiple of 4 or of a chunk, a draft
distribution close to the target (mostly accepted) and far from it (mostly rejected, several residual
steps per node), and a broken parent array.
"""
import numpy as np
import pytest
import torch

import oracle.sampling_oracle as so
from speculative_decoding_verify_decode_gb300 import native, synth

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _tree(seed, budget):
    return synth.ddtree_parents(np.random.default_rng(seed), budget)[0]


def _case(parents_list, V, T, seed, closeness):
    """Target logits, a draft distribution per node (softmax of the target logits plus noise of scale
    `closeness`, at the same temperature), drafts drawn from their parent's draft distribution, uniforms."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    indptr = np.concatenate([[0], np.cumsum([len(p) for p in parents_list])]).astype(np.int32)
    parents = np.concatenate(parents_list).astype(np.int32)
    n = int(indptr[-1])
    # a target row puts most of its mass on a few tokens: three spikes over N(0, 1) logits
    logits = torch.randn((n, V), generator=g, device="cuda")
    rows = torch.arange(n, device="cuda")
    for height in (16.0, 15.0, 14.0):
        logits[rows, torch.randint(0, V, (n,), generator=g, device="cuda")] += height
    noise = closeness * torch.randn((n, V), generator=g, device="cuda")
    q = torch.softmax((logits + noise) / T, dim=-1).contiguous()
    drafts = torch.zeros(n, dtype=torch.int64, device="cuda")
    for b in range(len(parents_list)):
        lo = int(indptr[b])
        for j in range(1, len(parents_list[b])):
            drafts[lo + j] = torch.multinomial(q[lo + int(parents[lo + j])], 1, generator=g)[0]
    r_acc = torch.rand(n, generator=g, device="cuda")
    r_smp = torch.rand(n, generator=g, device="cuda")
    return indptr, parents, logits.contiguous(), q, drafts.to(torch.int32), r_acc, r_smp


def _run(indptr, parents, logits, q, drafts, r_acc, r_smp, T, max_path=64):
    B = len(indptr) - 1
    V = logits.shape[1]
    ws = torch.empty(native.sd_sample_accept_workspace_size(indptr, V), dtype=torch.uint8, device="cuda")
    lens = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty((B, max_path), dtype=torch.int32, device="cuda")
    toks = torch.empty((B, max_path), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    par = torch.as_tensor(parents, device="cuda")
    native.sd_sample_accept(indptr, V, T, logits, q, par, drafts, r_acc, r_smp, lens, path, toks, max_path, ws,
                            status)
    torch.cuda.synchronize()
    return lens.cpu().numpy(), path.cpu().numpy(), toks.cpu().numpy(), int(status.item())


CASES = {
    # name: (parents per sequence, vocab, temperature, draft closeness)
    "chain8_full_vocab_close": ([synth.chain_parents(8)] * 4, 151936, 1.0, 0.3),
    "tree22_full_vocab_close": ([_tree(1, 22), _tree(2, 22)], 151936, 0.7, 0.3),
    "tree22_far_draft": ([_tree(3, 22), _tree(4, 30)], 151936, 1.0, 3.0),
    "ragged_hot": ([synth.chain_parents(0), _tree(5, 12), synth.chain_parents(3), synth.chain_parents(0)], 4099,
                   2.0, 0.5),
    "odd_vocab_cold": ([_tree(6, 16), synth.chain_parents(5)], 1001, 0.5, 1.0),
    "tiny_vocab_trees": ([_tree(7 + i, 10) for i in range(6)], 7, 1.0, 1.0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_sampling_verify_matches_oracle(name):
    parents_list, V, T, closeness = CASES[name]
    compared = total = 0
    for rep in range(3):
        indptr, parents, logits, q, drafts, r_acc, r_smp = _case(parents_list, V, T, 1000 * rep + len(name),
                                                                 closeness)
        lens, path, toks, status = _run(indptr, parents, logits, q, drafts, r_acc, r_smp, T)
        assert status == 0
        f64 = lambda t: t.detach().cpu().numpy().astype(np.float64)
        rl, rp, rt, margin = so.sampling_accept(indptr, parents, drafts.cpu().numpy(), f64(logits), f64(q), T,
                                                f64(r_acc), f64(r_smp))
        for b in range(len(indptr) - 1):
            total += 1
            a = int(lens[b])
            n = int(indptr[b + 1] - indptr[b])
            # always valid: a root path of accepted drafts, tokens in range, -1 padding
            assert 1 <= a <= n and path[b, 0] == 0 and (path[b, a:] == -1).all() and (toks[b, a:] == -1).all()
            for i in range(1, a):
                assert parents[indptr[b] + path[b, i]] == path[b, i - 1]
                assert toks[b, i - 1] == drafts[indptr[b] + path[b, i]].item()
            assert 0 <= toks[b, a - 1] < V
            if margin[b] > 5e-5:
                compared += 1
                assert a == rl[b], (b, a, rl[b])
                assert list(path[b, :a]) == list(rp[b])
                assert list(toks[b, :a]) == list(rt[b])
    assert compared >= 0.5 * total, (compared, total)


def test_broken_parents_keep_the_root():
    indptr, parents, logits, q, drafts, r_acc, r_smp = _case([_tree(20, 8)], 4096, 1.0, 20, 0.3)
    parents = parents.copy()
    parents[5] = 7                                  # a parent after its child
    lens, path, toks, status = _run(indptr, parents, logits, q, drafts, r_acc, r_smp, 1.0)
    assert status & native.SD_DEV_BAD_PARENTS
    assert lens[0] == 1 and path[0, 0] == 0 and 0 <= toks[0, 0] < 4096
