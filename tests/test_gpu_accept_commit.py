"""GPU argmax/accept and KV commit (through the C ABI) against the oracle.

Both must be bit-exact: target tokens, accept lengths, path node ids, emitted
tokens and every byte of every cache page.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_decode_gb300 import native, synth
from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs

from gpu_helpers import ensure_built, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _run_accept(w, logits, max_path=None):
    d = device_inputs(w)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, 1, logits.shape[1], max_path=max_path)
    st.accept(logits, d["parents"], d["draft_tokens"])
    torch.cuda.synchronize()
    return st


def _check_accept(w, logits, st):
    lg = logits.detach().cpu().numpy()
    t, lens, paths, toks = oracle.accept(w.q_indptr, w.parents, w.draft_tokens, lg)
    np.testing.assert_array_equal(st.target_tokens.cpu().numpy(), t)
    np.testing.assert_array_equal(st.accept_len.cpu().numpy(), lens)
    path = st.path.cpu().numpy()
    out = st.out_tokens.cpu().numpy()
    for b in range(w.batch):
        a = int(lens[b])
        assert list(path[b, :a]) == paths[b]
        assert list(out[b, :a]) == toks[b]
        assert (path[b, a:] == -1).all() and (out[b, a:] == -1).all()
    assert int(st.dev_status.item()) == 0
    return lens


@pytest.mark.parametrize("name", ["tiny_chain_ctx512", "chain8_ctx4k", "ddtree22_ctx32k",
                                  "conc8_chain4_ragged", "ddtree22_ctx128k"])
def test_accept_on_workloads(name):
    w = synth.make_workload(name, device="cuda", layers=0, ctx_override=16)
    st = _run_accept(w, w.logits)
    _check_accept(w, w.logits, st)


@pytest.mark.parametrize("vocab", [151936, 4096, 1001, 64])
def test_accept_unplanted_normal_logits(vocab):
    rng = np.random.default_rng(vocab)
    parents = [synth.ddtree_parents(rng, 22)[0], synth.chain_parents(8), synth.chain_parents(0)]
    w = workload(parents, [16, 16, 16], seed=3, vocab=vocab, logits=False)
    g = torch.Generator(device="cuda").manual_seed(vocab)
    logits = torch.randn((w.total_nodes, vocab), generator=g, device="cuda")
    t = logits.argmax(dim=1).cpu().numpy()          # plant drafts on the true argmax
    for b in range(w.batch):
        lo, hi = int(w.q_indptr[b]), int(w.q_indptr[b + 1])
        w.draft_tokens[lo:hi] = synth.plant_drafts(rng, w.parents[lo:hi], t[lo:hi], vocab, 0.8)
    st = _run_accept(w, logits)
    _check_accept(w, logits, st)


def test_vocab_of_one_accepts_every_draft():
    w = workload([synth.chain_parents(6)], [16], seed=5, vocab=1, p=1.0, logits=False)
    w.draft_tokens = np.zeros(7, dtype=np.int32)
    logits = torch.randn((7, 1), device="cuda")
    st = _run_accept(w, logits)
    lens = _check_accept(w, logits, st)
    assert lens[0] == 7


def test_argmax_ties_across_chunks_and_signed_zero():
    vocab = 151936
    w = workload([synth.chain_parents(7)], [16], seed=4, vocab=vocab, logits=False)
    logits = torch.randn((8, vocab), device="cuda").clamp_(-5, 5)
    logits[0, 9000] = logits[0, 5] = logits[0, 150000] = 7.0      # first index wins, across chunks
    logits[1, 4095] = logits[1, 4096] = 7.0                          # chunk boundary
    logits[2].zero_(); logits[2, 3] = -0.0                            # +0 / -0 compare equal
    logits[3].fill_(-0.0); logits[3, 0] = 0.0
    logits[4].fill_(-float("inf"))                                    # all -inf -> index 0
    logits[5].fill_(1.25)                                             # all equal -> index 0
    logits[6, 151935] = 9.0                                           # last element
    logits[7, 1000:1256] = 8.0                                        # 256 equal values in one chunk
    st = _run_accept(w, logits)
    _check_accept(w, logits, st)
    assert list(st.target_tokens.cpu().numpy()[:8]) == [5, 4095, 0, 0, 0, 0, 151935, 1000]


def test_duplicate_siblings_longest_then_lexicographic():
    vocab = 64
    # (parents, draft, target argmax per node) from the hand-worked cases
    cases = [([-1, 0, 0, 2], [1, 7, 7, 9], [7, 8, 9, 3]),
             ([-1, 0, 0, 1, 2], [1, 7, 7, 5, 5], [7, 5, 5, 30, 31]),
             ([-1, 0, 0, 1, 2, 4], [3, 60, 10, 11, 12, 14], [10, 11, 12, 13, 14, 15])]
    parents = [np.array(c[0], dtype=np.int32) for c in cases]
    w = workload(parents, [5, 6, 7], seed=8, vocab=vocab, logits=False)
    w.draft_tokens = np.concatenate([np.array(c[1], dtype=np.int32) for c in cases])
    logits = torch.zeros((w.total_nodes, vocab), device="cuda")
    t = np.concatenate([c[2] for c in cases])
    logits[torch.arange(w.total_nodes), torch.as_tensor(t, device="cuda")] = 1.0
    st = _run_accept(w, logits)
    lens = _check_accept(w, logits, st)
    assert list(lens) == [3, 3, 4]


def test_all_rejected_gives_one_token():
    vocab = 500
    rng = np.random.default_rng(11)
    par = synth.ddtree_parents(rng, 22)[0]
    w = workload([par], [16], seed=9, vocab=vocab, logits=False)
    logits = torch.randn((23, vocab), device="cuda")
    t = logits.argmax(dim=1).cpu().numpy()
    w.draft_tokens = np.array([(t[max(int(p), 0)] + 1) % vocab for p in par], dtype=np.int32)
    st = _run_accept(w, logits)
    lens = _check_accept(w, logits, st)
    assert lens[0] == 1 and int(st.out_tokens[0, 0]) == int(t[0])


def test_path_overflow_and_bad_parents_are_reported():
    w = workload([synth.chain_parents(8)], [16], seed=10, vocab=100, logits=False)
    logits = torch.zeros((9, 100), device="cuda")
    logits[:, 7] = 1.0
    w.draft_tokens = np.full(9, 7, dtype=np.int32)        # every draft accepted: A = 9
    st = _run_accept(w, logits, max_path=4)
    assert int(st.accept_len.item()) == 4
    assert int(st.dev_status.item()) & native.SD_DEV_PATH_OVERFLOW
    w.parents = np.array([-1, 0, 1, 5, 3, 4, 5, 6, 7], dtype=np.int32)   # node 3 points forward
    st = _run_accept(w, logits)
    assert int(st.dev_status.item()) & native.SD_DEV_BAD_PARENTS
    assert int(st.accept_len.item()) == 3                     # nodes 0..2 stay valid


# ---------------------------------------------------------------- commit

def _random_bits(shape, g):
    return torch.randint(-32768, 32767, shape, generator=g, device="cuda", dtype=torch.int16).view(torch.bfloat16)


def test_commit_matches_oracle_bytes():
    rng = np.random.default_rng(12)
    parents = [synth.chain_parents(4), synth.ddtree_parents(rng, 22)[0], synth.chain_parents(0),
               synth.chain_parents(8)]
    ctx = [31, 0, 16, 4090]
    w = synth.make_structure(4, ctx, parents, 12, 100, [0.8] * 4, spare_pages=5)
    layers = 3
    g = torch.Generator(device="cuda").manual_seed(12)
    kc = [_random_bits((w.num_pool_pages, 4, 16, 256), g) for _ in range(layers)]
    vc = [_random_bits((w.num_pool_pages, 4, 16, 256), g) for _ in range(layers)]
    kn = [_random_bits((w.total_nodes, 4, 256), g) for _ in range(layers)]
    vn = [_random_bits((w.total_nodes, 4, 256), g) for _ in range(layers)]
    lens = np.array([5, 4, 1, 2], dtype=np.int32)
    _, depth = oracle.tree_ancestors(parents[1])
    deep = int(np.flatnonzero(depth == 3)[0])
    p1, _ = oracle.tree_ancestors(parents[1])
    paths = [[0, 1, 2, 3, 4], p1[deep], [0], [0, 1]]
    max_path = 64
    path = np.full((4, max_path), -1, dtype=np.int32)
    for b, pth in enumerate(paths):
        path[b, :len(pth)] = pth
    ref_k, ref_v, ref_ctx = oracle.kv_commit([t.view(torch.int16).cpu().numpy() for t in kc],
                                             [t.view(torch.int16).cpu().numpy() for t in vc],
                                             [t.view(torch.int16).cpu().numpy() for t in kn],
                                             [t.view(torch.int16).cpu().numpy() for t in vn],
                                             w.page_table, w.ctx_lens, w.q_indptr, lens, paths)
    d = device_inputs(w)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, layers, 100, max_path=max_path)
    st.accept_len.copy_(torch.as_tensor(lens))
    st.path.copy_(torch.as_tensor(path))
    st.commit(kc, vc, kn, vn, d["page_table"], d["ctx_lens"])
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    np.testing.assert_array_equal(st.new_ctx_lens.cpu().numpy(), ref_ctx)
    for layer in range(layers):
        np.testing.assert_array_equal(kc[layer].view(torch.int16).cpu().numpy(), ref_k[layer])
        np.testing.assert_array_equal(vc[layer].view(torch.int16).cpu().numpy(), ref_v[layer])


def test_commit_rejects_bad_accept_and_leaves_cache():
    w = synth.make_structure(2, [20, 40], [synth.chain_parents(4)] * 2, 13, 100, [0.8] * 2)
    g = torch.Generator(device="cuda").manual_seed(13)
    kc = [_random_bits((w.num_pool_pages, 4, 16, 256), g)]
    vc = [_random_bits((w.num_pool_pages, 4, 16, 256), g)]
    kn = [_random_bits((w.total_nodes, 4, 256), g)]
    vn = [_random_bits((w.total_nodes, 4, 256), g)]
    k0, v0 = kc[0].clone(), vc[0].clone()
    d = device_inputs(w)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, 1, 100)
    st.accept_len.copy_(torch.tensor([2, 9], dtype=torch.int32))           # 9 > N = 5
    st.path.copy_(torch.tensor([[0, 7, -1, -1, -1], [0, 1, 2, 3, 4]], dtype=torch.int32))  # node 7 > N
    st.commit(kc, vc, kn, vn, d["page_table"], d["ctx_lens"])
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & native.SD_DEV_BAD_ACCEPT
    assert torch.equal(kc[0].view(torch.int16), k0.view(torch.int16))
    assert torch.equal(vc[0].view(torch.int16), v0.view(torch.int16))


def test_full_step_matches_oracle():
    """attention for every layer + accept + commit on a reduced chain workload."""
    w = synth.make_workload("chain8_ctx4k", device="cuda", layers=3, ctx_override=777)
    d = device_inputs(w)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, w.layers, w.vocab)
    kc0 = [t.clone() for t in w.k_cache]
    vc0 = [t.clone() for t in w.v_cache]
    st.run(w.q, w.k_cache, w.v_cache, w.k_new, w.v_new, d["page_table"], d["ctx_lens"], d["parents"],
           d["draft_tokens"], w.logits)
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    t, lens, paths, toks = oracle.accept(w.q_indptr, w.parents, w.draft_tokens, w.logits.cpu().numpy())
    assert list(st.accept_len.cpu().numpy()) == list(lens)
    u16 = lambda ts: [x.view(torch.int16).cpu().numpy() for x in ts]
    ref_k, ref_v, ref_ctx = oracle.kv_commit(u16(kc0), u16(vc0), u16(w.k_new), u16(w.v_new), w.page_table,
                                             w.ctx_lens, w.q_indptr, lens, paths)
    for layer in range(w.layers):
        np.testing.assert_array_equal(u16([w.k_cache[layer]])[0], ref_k[layer])
        np.testing.assert_array_equal(u16([w.v_cache[layer]])[0], ref_v[layer])
    np.testing.assert_array_equal(st.new_ctx_lens.cpu().numpy(), ref_ctx)
