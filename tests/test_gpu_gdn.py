"""Tree Gated DeltaNet on the GPU, through the C ABI, against the oracle.

The short convolution along the parent chain (every channel, trees, ragged batch, a channel count that is not
a multiple of the block), the gated delta rule over the tree (element by element, small and full head
geometry, N = 1 .. 64, chains, strong decay that underflows the path products), and persist-on-accept of
the recurrent state (fp32, every layer in one launch) and of the convolution state (bytes); an out-of-range
accept result leaves the states untouched.
"""
import numpy as np
import pytest
import torch

import oracle.gdn_oracle as gd
from speculative_decoding_verify_decode_gb300 import native, synth

from gpu_helpers import ensure_built, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _tree(seed, budget):
    return synth.ddtree_parents(np.random.default_rng(seed), budget)[0]


def _batch(parents_list):
    indptr = np.concatenate([[0], np.cumsum([len(p) for p in parents_list])]).astype(np.int32)
    parents = np.concatenate(parents_list).astype(np.int32)
    return indptr, parents


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device="cuda")


def _run_tree(parents_list, seed, hk, hv, decay=0.5):
    indptr, parents = _batch(parents_list)
    x = synth.gdn_inputs(int(indptr[-1]), len(parents_list), seed, device="cuda", hk=hk, hv=hv, channels=8,
                         decay=decay)
    shape = native.GdnShape(indptr, hk, hv)
    cache = torch.empty(native.sd_gdn_tree_cache_size(shape), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x.v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.sd_gdn_tree(shape, x.q, x.k, x.v, x.g, x.beta, x.state, _i32(parents), out, cache, status)
    torch.cuda.synchronize()
    return indptr, parents, x, shape, cache, out, int(status.item())


def _oracle_tree(indptr, parents, x):
    return gd.gdn_tree(f64(x.q), f64(x.k), f64(x.v), f64(x.g), f64(x.beta), f64(x.state), indptr, parents)


TREES = {
    "tree22": ([_tree(1, 22)], 2, 4),
    "chain9_and_tree": ([synth.chain_parents(8), _tree(2, 14)], 2, 4),
    "ragged_batch": ([synth.chain_parents(0), _tree(3, 22), synth.chain_parents(4), _tree(4, 63)], 1, 2),
    "full_heads_tree22": ([_tree(5, 22)], 16, 32),
}


@pytest.mark.parametrize("name", sorted(TREES))
def test_gdn_tree_matches_oracle(name):
    parents_list, hk, hv = TREES[name]
    indptr, parents, x, _, _, out, status = _run_tree(parents_list, len(name), hk, hv)
    assert status == 0
    ref, _ = _oracle_tree(indptr, parents, x)
    got = f64(out)
    err = float(np.abs(got - ref).max())
    assert np.isfinite(got).all()
    assert err <= 1e-2 * float(np.abs(ref).max()) + 1e-6, err


def test_strong_decay_underflowing_path_products():
    indptr, parents, x, _, _, out, status = _run_tree([_tree(6, 40)], 6, 2, 4, decay=60.0)
    assert status == 0
    ref, _ = _oracle_tree(indptr, parents, x)
    got = f64(out)
    assert np.isfinite(got).all()
    assert float(np.abs(got - ref).max()) <= 1e-2 * float(np.abs(ref).max()) + 1e-6


def _root_path(parents, lo, j):
    out = []
    u = j
    while u >= 0:
        out.append(u)
        u = int(parents[lo + u])
    return out[::-1]


def test_commit_of_state_and_convolution_every_layer():
    parents_list = [_tree(7, 22), synth.chain_parents(6), _tree(8, 30)]
    indptr, parents = _batch(parents_list)
    n, B, hk, hv, C = int(indptr[-1]), len(parents_list), 2, 4, 300
    shape = native.GdnShape(indptr, hk, hv)
    rng = np.random.default_rng(9)
    last = [int(rng.integers(0, len(p))) for p in parents_list]
    paths = [_root_path(parents, int(indptr[b]), last[b]) for b in range(B)]
    max_path = 64
    path_arr = np.full((B, max_path), -1, dtype=np.int32)
    for b, pth in enumerate(paths):
        path_arr[b, :len(pth)] = pth
    lens = np.array([len(pth) for pth in paths], dtype=np.int32)
    layers, caches, states0, conv0, xs = [], [], [], [], []
    for layer in range(3):
        x = synth.gdn_inputs(n, B, 20 + layer, device="cuda", hk=hk, hv=hv, channels=C)
        cache = torch.empty(native.sd_gdn_tree_cache_size(shape), dtype=torch.uint8, device="cuda")
        out = torch.empty_like(x.v)
        native.sd_gdn_tree(shape, x.q, x.k, x.v, x.g, x.beta, x.state, _i32(parents), out, cache)
        layers.append(x)
        caches.append(cache)
        states0.append(f64(x.state))
        conv0.append(x.conv_state.clone())
        xs.append(x.x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.sd_gdn_commit(shape, [x.state for x in layers], caches, _i32(lens), _i32(path_arr),
                         conv_state_layers=[x.conv_state for x in layers], x_layers=xs, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for layer, x in enumerate(layers):
        _, node_states = gd.gdn_tree(f64(x.q), f64(x.k), f64(x.v), f64(x.g), f64(x.beta), states0[layer], indptr,
                                     parents)
        ref = gd.gdn_commit(states0[layer], node_states, indptr, lens, paths)
        got = f64(x.state)
        assert float(np.abs(got - ref).max()) <= 2e-4 * float(np.abs(ref).max()) + 1e-6
        u16 = lambda t: t.view(torch.int16).cpu().numpy()
        ref_conv = gd.conv_commit(u16(conv0[layer]), u16(xs[layer]), indptr, lens, paths)
        np.testing.assert_array_equal(u16(x.conv_state), ref_conv)


def test_bad_accept_leaves_states_untouched():
    parents_list = [_tree(10, 10)]
    indptr, parents, x, shape, cache, _, _ = _run_tree(parents_list, 10, 2, 4)
    before = x.state.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    path = _i32(np.array([[0, 1, 2, 3]]))
    native.sd_gdn_commit(shape, [x.state], [cache], _i32(np.array([40])), path, dev_status=status)   # A > N
    torch.cuda.synchronize()
    assert int(status.item()) & native.SD_DEV_BAD_ACCEPT
    assert torch.equal(before, x.state)


CONV = {
    "tree22_full_channels": ([_tree(11, 22)], synth.GDN_CHANNELS),
    "ragged_odd_channels": ([synth.chain_parents(0), _tree(12, 9), synth.chain_parents(2), _tree(13, 63)], 300),
}


@pytest.mark.parametrize("name", sorted(CONV))
def test_conv_tree_matches_oracle(name):
    parents_list, C = CONV[name]
    indptr, parents = _batch(parents_list)
    x = synth.gdn_inputs(int(indptr[-1]), len(parents_list), 30 + len(name), device="cuda", hk=1, hv=1, channels=C)
    y = torch.empty_like(x.x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.sd_gdn_conv_tree(indptr, x.x, x.conv_w, x.conv_state, _i32(parents), y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = gd.conv_tree(f64(x.x), f64(x.conv_w), f64(x.conv_state), indptr, parents)
    err = float(np.abs(f64(y) - ref).max())
    assert err <= 1e-2 * float(np.abs(ref).max()) + 1e-5, err
