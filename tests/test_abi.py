"""The C ABI without a GPU: the library builds, loads, exports every symbol
the header declares, and rejects bad host-side arguments before any launch.

Every call below fails a host check, so no kernel is ever launched with the
placeholder pointers used here.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from speculative_decoding_verify_decode_gb300 import build, native

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = [os.path.join(INCLUDE, f) for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h")]
FAKE = 0x10000   # never dereferenced: each call returns before launching


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def test_every_declared_symbol_is_exported(lib):
    names = set()
    for h in HEADERS:
        names |= set(re.findall(r"\b(sd_[a-z0-9_]+)\s*\(", open(h).read()))
    assert {"sd_verify_attn", "sd_accept", "sd_kv_commit", "sd_status_string", "sd_verify_attn_fp8",
            "sd_kv_commit_fp8", "sd_gdn_tree", "sd_gdn_commit", "sd_gdn_conv_tree", "sd_sample_accept"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert native.status_string(0) == "ok"
    assert "workspace" in native.status_string(4)


def _shape(indptr=(0, 5), **kw):
    s = native.Shape(list(indptr), kw.pop("max_pages", 40), kw.pop("pool", 40), kw.pop("splits", 0))
    for k, v in kw.items():
        setattr(s.c, k, v)
    return s


def _attn(lib, shape, ws=None, ws_bytes=0, q=FAKE):
    return lib.sd_verify_attn(shape.ref, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, ws, ws_bytes,
                              None, None)


def test_geometry_other_than_24_4_256_16_is_unsupported(lib):
    for field, bad in [("num_q_heads", 32), ("num_kv_heads", 8), ("head_dim", 128), ("page_size", 64)]:
        assert _attn(lib, _shape(**{field: bad})) == native.SD_ERR_UNSUPPORTED
        assert lib.sd_verify_attn_workspace_size(_shape(**{field: bad}).ref) == 0


def test_node_counts(lib):
    assert _attn(lib, _shape((0, 65))) == native.SD_ERR_UNSUPPORTED        # N > 64
    assert _attn(lib, _shape((0, 5, 5))) == native.SD_ERR_INVALID_ARG      # N = 0
    assert _attn(lib, _shape((1, 5))) == native.SD_ERR_INVALID_ARG         # indptr[0] != 0
    s = _shape()
    s.c.batch = 0
    assert _attn(lib, s) == native.SD_ERR_INVALID_ARG
    s.c.batch = native.MAX_BATCH + 1
    assert _attn(lib, s) == native.SD_ERR_INVALID_ARG


def test_null_pointers_and_workspace(lib):
    assert _attn(lib, _shape(), q=None) == native.SD_ERR_INVALID_ARG
    big = _shape((0, 23), max_pages=2050, pool=2050)
    need = lib.sd_verify_attn_workspace_size(big.ref)
    assert need > 0
    assert _attn(lib, big, ws=None, ws_bytes=0) == native.SD_ERR_WORKSPACE
    assert _attn(lib, big, ws=FAKE, ws_bytes=need - 1) == native.SD_ERR_WORKSPACE


def test_misaligned_tensors_rejected(lib):
    assert _attn(lib, _shape(), q=FAKE + 8) == native.SD_ERR_INVALID_ARG
    s = _shape()
    arr = (ctypes.c_void_p * 1)(FAKE + 2)
    ok = (ctypes.c_void_p * 1)(FAKE)
    assert lib.sd_kv_commit(s.ref, 1, arr, ok, ok, ok, FAKE, FAKE, None, FAKE, FAKE, 8, None, None) \
        == native.SD_ERR_INVALID_ARG


def test_workspace_grows_with_context_and_nodes(lib):
    a = lib.sd_verify_attn_workspace_size(_shape((0, 9), max_pages=257, pool=257).ref)
    b = lib.sd_verify_attn_workspace_size(_shape((0, 23), max_pages=8194, pool=8194).ref)
    assert b > a


def test_accept_host_checks(lib):
    ind = (ctypes.c_int * 2)(0, 23)
    need = lib.sd_accept_workspace_size(1, ind, 151936)
    assert need >= 23 * 38 * 8
    call = lambda vocab, max_path, ws, ws_bytes, logits=FAKE: lib.sd_accept(
        1, ind, vocab, logits, FAKE, FAKE, FAKE, FAKE, FAKE, None, max_path, ws, ws_bytes, None, None)
    assert call(0, 17, FAKE, need) == native.SD_ERR_INVALID_ARG
    assert call(151936, 0, FAKE, need) == native.SD_ERR_INVALID_ARG
    assert call(151936, 17, FAKE, need, logits=None) == native.SD_ERR_INVALID_ARG
    assert call(151936, 17, FAKE, need - 1) == native.SD_ERR_WORKSPACE
    assert call(151936, 17, None, 0) == native.SD_ERR_WORKSPACE


def test_commit_host_checks(lib):
    s = _shape()
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    nul = (ctypes.c_void_p * 2)(FAKE, None)
    call = lambda layers, k=arr, new=None, ctx=FAKE: lib.sd_kv_commit(
        s.ref, layers, k, arr, arr, arr, FAKE, ctx, new, FAKE, FAKE, 8, None, None)
    assert call(0) == native.SD_ERR_INVALID_ARG
    assert call(native.MAX_LAYERS + 1) == native.SD_ERR_UNSUPPORTED
    assert call(2, k=nul) == native.SD_ERR_INVALID_ARG
    assert call(2, new=FAKE, ctx=FAKE) == native.SD_ERR_INVALID_ARG   # new_ctx_lens aliases ctx_lens


def test_ddtree_host_checks(lib):
    ws = FAKE
    call = lambda b, p, v, k, n, ws_bytes=1 << 30, logits=FAKE: lib.sd_ddtree_build(
        b, p, v, k, n, logits, FAKE, FAKE, FAKE, None, ws, ws_bytes, None, None)
    assert call(1, 16, 151936, 9, 22) == native.SD_ERR_UNSUPPORTED        # topk > 8
    assert call(1, 65, 151936, 8, 22) == native.SD_ERR_UNSUPPORTED        # positions > 64
    assert call(1, 16, 151936, 8, 64) == native.SD_ERR_UNSUPPORTED        # 1 + budget > 64
    assert call(0, 16, 151936, 8, 22) == native.SD_ERR_INVALID_ARG
    assert call(1, 16, 4, 8, 22) == native.SD_ERR_INVALID_ARG             # vocab < topk
    assert call(1, 16, 151936, 8, 22, logits=None) == native.SD_ERR_INVALID_ARG
    assert call(1, 16, 151936, 8, 22, ws_bytes=16) == native.SD_ERR_WORKSPACE
    assert lib.sd_ddtree_workspace_size(1, 16, 151936, 8) > 0
    assert lib.sd_ddtree_workspace_size(1, 16, 151936, 9) == 0


def test_negative_window_is_rejected(lib):
    s = _shape()
    s.c.window = -1
    assert _attn(lib, s) == native.SD_ERR_INVALID_ARG
    assert lib.sd_verify_attn_workspace_size(s.ref) == 0


def test_fp8_scales_checked_before_any_launch(lib):
    s = _shape()
    attn = lambda ks, vs, kc=FAKE: lib.sd_verify_attn_fp8(s.ref, FAKE, kc, FAKE, ks, vs, FAKE, FAKE, FAKE, FAKE,
                                                          FAKE, FAKE, None, None, 0, None, None)
    for bad in (0.0, -1.0, float("inf"), float("nan"), 1e-45):     # 1e-45: the reciprocal overflows fp32
        assert attn(bad, 1.0) == native.SD_ERR_INVALID_ARG, bad
        assert attn(1.0, bad) == native.SD_ERR_INVALID_ARG, bad
    assert attn(1.0, 1.0, kc=FAKE + 4) == native.SD_ERR_INVALID_ARG   # codes must start on 16 bytes
    assert attn(1.0, 1.0, kc=None) == native.SD_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    good = (ctypes.c_float * 2)(0.5, 0.25)
    bad = (ctypes.c_float * 2)(0.5, 0.0)
    commit = lambda ks, vs: lib.sd_kv_commit_fp8(s.ref, 2, arr, arr, ks, vs, arr, arr, FAKE, FAKE, None, FAKE,
                                                 FAKE, 8, None, None)
    assert commit(None, good) == native.SD_ERR_INVALID_ARG
    assert commit(good, bad) == native.SD_ERR_INVALID_ARG
    assert commit(bad, good) == native.SD_ERR_INVALID_ARG



def test_gdn_host_checks(lib):
    ind = [0, 23]
    ok = native.GdnShape(ind, 16, 32)
    assert lib.sd_gdn_tree_cache_size(ok.ref) == 23 * 32 * 128 * 4 + 3072 + 23 * 16 * 128 * 4
    assert lib.sd_gdn_tree_cache_size(native.GdnShape(ind, 16, 32, head_dim=64).ref) == 0
    assert lib.sd_gdn_tree_cache_size(native.GdnShape(ind, 16, 24).ref) == 0      # H_v not a multiple of H_k
    call = lambda s, cache=FAKE, nbytes=1 << 30, q=FAKE: lib.sd_gdn_tree(s.ref, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                                        FAKE, cache, nbytes, None, None)
    assert call(native.GdnShape(ind, 16, 32, head_dim=256)) == native.SD_ERR_UNSUPPORTED
    assert call(native.GdnShape(ind, 16, 512)) == native.SD_ERR_UNSUPPORTED
    assert call(native.GdnShape(ind, 0, 32)) == native.SD_ERR_INVALID_ARG
    assert call(ok, q=None) == native.SD_ERR_INVALID_ARG
    assert call(ok, q=FAKE + 2) == native.SD_ERR_INVALID_ARG
    assert call(ok, cache=None) == native.SD_ERR_WORKSPACE
    assert call(ok, nbytes=16) == native.SD_ERR_WORKSPACE
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    commit = lambda layers, ch=0, conv=None: lib.sd_gdn_commit(ok.ref, layers, arr, arr, ch, conv, conv, FAKE, FAKE,
                                                               8, None, None)
    assert commit(0) == native.SD_ERR_INVALID_ARG
    assert commit(native.MAX_LAYERS + 1) == native.SD_ERR_UNSUPPORTED
    assert commit(2, ch=8192, conv=None) == native.SD_ERR_INVALID_ARG
    ind2 = (ctypes.c_int * 2)(0, 23)
    assert lib.sd_gdn_conv_tree(1, ind2, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == native.SD_ERR_INVALID_ARG
    assert lib.sd_gdn_conv_tree(1, ind2, 64, None, FAKE, FAKE, FAKE, FAKE, None, None) == native.SD_ERR_INVALID_ARG


def test_sample_accept_host_checks(lib):
    ind = (ctypes.c_int * 2)(0, 23)
    need = lib.sd_sample_accept_workspace_size(1, ind, 151936)
    assert need >= 23 * 38 * 8
    call = lambda vocab, t, ws=FAKE, nbytes=need, logits=FAKE: lib.sd_sample_accept(
        1, ind, vocab, t, logits, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 17, ws, nbytes, None, None)
    for bad_t in (0.0, -1.0, float("inf"), float("nan"), 1e-45):
        assert call(151936, bad_t) == native.SD_ERR_INVALID_ARG, bad_t
    assert call(0, 1.0) == native.SD_ERR_INVALID_ARG
    assert call(2048 * 1024 + 1, 1.0) == native.SD_ERR_UNSUPPORTED
    assert call(151936, 1.0, logits=None) == native.SD_ERR_INVALID_ARG
    assert call(151936, 1.0, ws=None) == native.SD_ERR_WORKSPACE
    assert call(151936, 1.0, nbytes=need - 1) == native.SD_ERR_WORKSPACE
