"""sd_verify_attn_noalloc: the entry point for callers that cannot allocate
device memory (a plugin whose device memory belongs to another runtime's
pool, or a loop where allocating is not allowed).  It must give the same
attention output as sd_verify_attn with a caller workspace, call after call,
while its scratch lives in one fixed array inside the library.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verify_decode_gb300 import native, synth
from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs

from gpu_helpers import ensure_built, f64, tight_bound


def _attn_args(w, layer=0):
    d = device_inputs(w)
    return (w.q[layer], w.k_cache[layer], w.v_cache[layer], w.k_new[layer], w.v_new[layer], d["page_table"],
            d["ctx_lens"], d["parents"])


def test_invalid_shape_returns_the_shape_status():
    ensure_built()
    shape = native.Shape(np.array([0, 9]), 64, 64)
    shape.c.head_dim = 128                       # geometry the library does not support
    with pytest.raises(native.SdError) as e:
        native.sd_verify_attn_noalloc(shape, 16, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)   # never dereferenced
    assert e.value.status == native.SD_ERR_UNSUPPORTED


def test_oversized_shape_is_rejected_before_any_launch():
    ensure_built()
    # 4 sequences of 64 nodes cut into 64 splits each need far more than the fixed scratch
    shape = native.Shape(np.arange(0, 5 * 64, 64), 8192, 8192 * 4, num_splits=64)
    assert native.sd_verify_attn_workspace_size(shape) > native.NOALLOC_SCRATCH_BYTES
    with pytest.raises(native.SdError) as e:
        native.sd_verify_attn_noalloc(shape, 16, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)   # never dereferenced
    assert e.value.status == native.SD_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["ddtree22_ctx32k", "conc8_chain4_ragged"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    w = synth.make_workload(name, device="cuda", layers=2, logits=False, qkv_scale=0.5)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, 1, 16, want_lse=True)
    assert 0 < native.sd_verify_attn_workspace_size(st.shape) <= native.NOALLOC_SCRATCH_BYTES
    for layer in (0, 1):          # two calls in a row share (and reuse) the scratch array
        args = _attn_args(w, layer)
        st.attention(0, *args)
        out = torch.empty_like(st.out[0])
        lse = torch.empty_like(st.lse[0])
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        native.sd_verify_attn_noalloc(st.shape, *args, out, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(st.dev_status.item()) == 0
        ref = f64(st.out[0])
        err = float(np.abs(f64(out) - ref).max())
        assert err <= tight_bound(ref), err
        assert float(np.abs(f64(lse) - f64(st.lse[0])).max()) <= 1e-5


@pytest.mark.gpu
def test_calls_after_the_first_leave_free_device_memory_unchanged():
    """The first call in a context may load the library's module (and with it the scratch array);
    every later call allocates nothing: free device memory stays the same, byte for byte."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    w = synth.make_workload("ddtree22_ctx32k", device="cuda", layers=1, logits=False)
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, 1, 16)
    args = _attn_args(w, 0)
    out = torch.empty_like(st.out[0])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.sd_verify_attn_noalloc(st.shape, *args, out, None, status)   # warm-up: may load the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        native.sd_verify_attn_noalloc(st.shape, *args, out, None, status)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert int(status.item()) == 0
