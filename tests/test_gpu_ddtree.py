"""GPU draft-tree construction (through the C ABI) against the oracle.

Trees (parents, tokens) are compared exactly wherever every best-first
decision of the oracle wins by more than the fp32 log-sum-exp error (the
oracle reports that margin; equal scores are ordered by creation on both
sides); scores within 1e-4.  Cases: K = 1 chains, K = 8 at the page's shape
(16 positions, budget 22, vocabulary 151936), ragged last chunks, a
vocabulary that is not a multiple of 4, tied logits across chunks, a batch,
a budget larger than the candidates, and NaN reporting.
"""
import numpy as np
import pytest
import torch

import oracle.ddtree_oracle as dd
from speculative_decoding_verify_decode_gb300 import native, synth

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

MARGIN = 1e-3    # fp32 log-sum-exp over <= 2^18 terms is good to ~1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _gpu(logits, topk, budget, roots):
    b, pos, vocab = logits.shape
    x = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    r = torch.tensor(roots, dtype=torch.int32, device="cuda")
    par = torch.empty((b, 1 + budget), dtype=torch.int32, device="cuda")
    tok = torch.empty_like(par)
    sc = torch.empty((b, 1 + budget), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(native.sd_ddtree_workspace_size(b, pos, vocab, topk), 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.sd_ddtree_build(x, topk, budget, r, par, tok, sc, ws, st)
    torch.cuda.synchronize()
    return par.cpu().numpy(), tok.cpu().numpy(), sc.cpu().numpy(), int(st.item())


CASES = {
    # name: (batch, positions, vocab, topk, budget, ties); the seed is len(name) unless SEEDS says otherwise
    "k1_chain": (2, 16, 5000, 1, 15, False),
    "k8_page_shape": (1, 16, 151936, 8, 22, False),
    "k8_budget63": (1, 16, 20000, 8, 63, False),
    "k4_ragged_chunk": (3, 9, 4096 * 3 + 100, 4, 30, False),
    "k6_vocab_not_mult4": (2, 12, 9999, 6, 40, False),
    "k8_small_vocab": (2, 5, 37, 8, 20, False),
    "k3_ties": (2, 8, 10000, 3, 25, True),
    "budget_above_candidates": (1, 3, 500, 2, 20, False),
    "batch8": (8, 16, 32000, 8, 22, False),
}
SEEDS = {"k8_small_vocab": 15}   # a seed whose best-first decisions are all clear of fp32 rounding


@pytest.mark.parametrize("name", sorted(CASES))
def test_ddtree_matches_oracle(name):
    batch, pos, vocab, topk, budget, ties = CASES[name]
    logits = synth.draft_logits(batch, pos, vocab, seed=SEEDS.get(name, len(name)), ties=ties)
    roots = list(range(100, 100 + batch))
    par, tok, sc, status = _gpu(logits, topk, budget, roots)
    assert status == 0
    for b in range(batch):
        rp, rt, rs, margin = dd.ddtree(logits[b], topk, budget, roots[b])
        n = len(rp)
        assert margin > MARGIN, "seeded inputs must not leave a near-tie"
        np.testing.assert_array_equal(par[b, :n], rp)
        np.testing.assert_array_equal(tok[b, :n], rt)
        np.testing.assert_allclose(sc[b, :n], rs, atol=1e-4, rtol=0)
        assert (par[b, n:] == -1).all() and (tok[b, n:] == -1).all()


def test_nan_logits_are_reported():
    logits = synth.draft_logits(1, 4, 5000, seed=3)
    logits[0, 2, 4321] = np.nan
    _, _, _, status = _gpu(logits, 4, 10, [1])
    assert status & native.SD_DEV_NAN_LOGITS
