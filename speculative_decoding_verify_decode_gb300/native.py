"""ctypes binding of libsdverify.so (include/sd_verify.h).

Argument marshalling only: every function here turns torch tensors into the
device pointers and host arrays of the C ABI and raises on a non-zero status.
All computation happens in the library's CUDA kernels.  There is no fallback:
if the library is missing or was not built for this GPU, the first call
raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdverify.so")

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED, SD_ERR_CUDA, SD_ERR_WORKSPACE = range(5)
SD_DEV_BAD_PARENTS = 1
SD_DEV_BAD_PAGE = 2
SD_DEV_BAD_CTX = 4
SD_DEV_BAD_ACCEPT = 8
SD_DEV_NAN_LOGITS = 16
SD_DEV_PATH_OVERFLOW = 32
SD_DEV_TIMEOUT = 64
MAX_NODES = 64
MAX_BATCH = 256
MAX_LAYERS = 64


class SdShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("q_indptr_h", ctypes.POINTER(ctypes.c_int)),
                ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("page_size", ctypes.c_int),
                ("max_pages_per_seq", ctypes.c_int), ("num_pool_pages", ctypes.c_int),
                ("num_splits", ctypes.c_int),
                ("window", ctypes.c_int), ("ctx_stable", ctypes.c_int)]


class SdGdnShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("q_indptr_h", ctypes.POINTER(ctypes.c_int)),
                ("num_k_heads", ctypes.c_int), ("num_v_heads", ctypes.c_int), ("head_dim", ctypes.c_int)]


class SdError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def load() -> ctypes.CDLL:
    """Load (once) and type the library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m speculative_decoding_verify_decode_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ip, fp, sz = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.c_void_p, ctypes.c_size_t
    shp = ctypes.POINTER(SdShape)
    lib.sd_status_string.restype = ctypes.c_char_p
    lib.sd_status_string.argtypes = [ctypes.c_int]
    lib.sd_verify_attn_workspace_size.restype = sz
    lib.sd_verify_attn_workspace_size.argtypes = [shp]
    lib.sd_verify_attn.restype = ctypes.c_int
    lib.sd_verify_attn.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, vp, fp, vp, sz, vp, vp]
    lib.sd_verify_attn_fp8.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.sd_verify_attn_fp8.argtypes = [shp, vp, vp, vp, f32, f32, vp, vp, vp, vp, vp, vp, fp, vp, sz, vp, vp]
    lib.sd_verify_attn_noalloc.restype = ctypes.c_int
    lib.sd_verify_attn_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, vp, fp, vp, vp]
    lib.sd_accept_workspace_size.restype = sz
    lib.sd_accept_workspace_size.argtypes = [ctypes.c_int, ip, ctypes.c_int]
    lib.sd_accept.restype = ctypes.c_int
    lib.sd_accept.argtypes = [ctypes.c_int, ip, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                              vp, sz, vp, vp]
    lib.sd_sample_accept_workspace_size.restype = sz
    lib.sd_sample_accept_workspace_size.argtypes = [ctypes.c_int, ip, ctypes.c_int]
    lib.sd_sample_accept.restype = ctypes.c_int
    lib.sd_sample_accept.argtypes = [ctypes.c_int, ip, ctypes.c_int, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp,
                                     vp, ctypes.c_int, vp, sz, vp, vp]
    lib.sd_kv_commit.restype = ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    lib.sd_kv_commit.argtypes = [shp, ctypes.c_int, pp, pp, pp, pp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp]
    lib.sd_kv_commit_fp8.restype = ctypes.c_int
    fpp = ctypes.POINTER(ctypes.c_float)
    lib.sd_kv_commit_fp8.argtypes = [shp, ctypes.c_int, pp, pp, fpp, fpp, pp, pp, vp, vp, vp, vp, vp, ctypes.c_int,
                                     vp, vp]
    gshp = ctypes.POINTER(SdGdnShape)
    lib.sd_gdn_tree_cache_size.restype = sz
    lib.sd_gdn_tree_cache_size.argtypes = [gshp]
    lib.sd_gdn_conv_tree.restype = ctypes.c_int
    lib.sd_gdn_conv_tree.argtypes = [ctypes.c_int, ip, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp]
    lib.sd_gdn_tree.restype = ctypes.c_int
    lib.sd_gdn_tree.argtypes = [gshp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.sd_gdn_commit.restype = ctypes.c_int
    lib.sd_gdn_commit.argtypes = [gshp, ctypes.c_int, pp, pp, ctypes.c_int, pp, pp, vp, vp, ctypes.c_int, vp, vp]
    lib.sd_ddtree_workspace_size.restype = sz
    lib.sd_ddtree_workspace_size.argtypes = [ctypes.c_int] * 4
    lib.sd_ddtree_build.restype = ctypes.c_int
    lib.sd_ddtree_build.argtypes = [ctypes.c_int] * 5 + [vp, vp, vp, vp, vp, vp, sz, vp, vp]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().sd_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != SD_OK:
        raise SdError(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the verify library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _indptr(q_indptr) -> ctypes.Array:
    arr = np.ascontiguousarray(np.asarray(q_indptr, dtype=np.int32))
    return (ctypes.c_int * len(arr))(*arr.tolist())


class Shape:
    """An sd_shape with its host q_indptr kept alive."""

    def __init__(self, q_indptr, max_pages_per_seq: int, num_pool_pages: int, num_splits: int = 0,
                 window: int = 0, ctx_stable: bool = False):
        self.indptr = _indptr(q_indptr)
        self.c = SdShape(len(self.indptr) - 1, ctypes.cast(self.indptr, ctypes.POINTER(ctypes.c_int)),
                         24, 4, 256, 16, int(max_pages_per_seq), int(num_pool_pages), int(num_splits),
                         int(window), int(bool(ctx_stable)))

    def with_ctx_stable(self, ctx_stable: bool = True) -> "Shape":
        """The same shape with the context-stable launch flag set (see sd_shape.ctx_stable)."""
        c = self.c
        return Shape(list(self.indptr), c.max_pages_per_seq, c.num_pool_pages, c.num_splits, c.window,
                     ctx_stable)

    @property
    def ref(self):
        return ctypes.byref(self.c)


def sd_verify_attn_workspace_size(shape: Shape) -> int:
    return int(load().sd_verify_attn_workspace_size(shape.ref))


def sd_verify_attn(shape: Shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, out,
                   lse=None, workspace=None, dev_status=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sd_verify_attn(shape.ref, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                 _ptr(page_table), _ptr(ctx_lens), _ptr(parents), _ptr(out), _ptr(lse),
                                 _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
           "sd_verify_attn")


def sd_verify_attn_fp8(shape: Shape, q, k_cache, v_cache, k_scale: float, v_scale: float, k_new, v_new,
                       page_table, ctx_lens, parents, out, lse=None, workspace=None, dev_status=None,
                       stream=None) -> None:
    """sd_verify_attn over e4m3 caches (uint8 [pool, 4, 16, 256]) with per-tensor scales."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sd_verify_attn_fp8(shape.ref, _ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                     float(v_scale), _ptr(k_new), _ptr(v_new), _ptr(page_table), _ptr(ctx_lens),
                                     _ptr(parents), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                     _ptr(dev_status), _stream(stream)),
           "sd_verify_attn_fp8")


NOALLOC_SCRATCH_BYTES = 16 << 20


def sd_verify_attn_noalloc(shape: Shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, out,
                           lse=None, dev_status=None, stream=None) -> None:
    """sd_verify_attn with the library's fixed scratch array instead of a caller workspace."""
    _check(load().sd_verify_attn_noalloc(shape.ref, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new),
                                         _ptr(v_new), _ptr(page_table), _ptr(ctx_lens), _ptr(parents), _ptr(out),
                                         _ptr(lse), _ptr(dev_status), _stream(stream)),
           "sd_verify_attn_noalloc")


def sd_accept_workspace_size(q_indptr, vocab: int) -> int:
    ind = _indptr(q_indptr)
    return int(load().sd_accept_workspace_size(len(ind) - 1, ind, int(vocab)))


def sd_accept(q_indptr, vocab: int, logits, parents, draft_tokens, accept_len, path, out_tokens,
              target_tokens=None, max_path: int | None = None, workspace=None, dev_status=None,
              stream=None) -> None:
    ind = _indptr(q_indptr)
    if max_path is None:
        max_path = path.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sd_accept(len(ind) - 1, ind, int(vocab), _ptr(logits), _ptr(parents), _ptr(draft_tokens),
                            _ptr(accept_len), _ptr(path), _ptr(out_tokens), _ptr(target_tokens),
                            int(max_path), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
           "sd_accept")


def sd_sample_accept_workspace_size(q_indptr, vocab: int) -> int:
    ind = _indptr(q_indptr)
    return int(load().sd_sample_accept_workspace_size(len(ind) - 1, ind, int(vocab)))


def sd_sample_accept(q_indptr, vocab: int, temperature: float, logits, draft_probs, parents, draft_tokens, r_accept,
                     r_sample, accept_len, path, out_tokens, max_path: int | None = None, workspace=None,
                     dev_status=None, stream=None) -> None:
    """Sampling-based verification at temperature T (speculative sampling, multi-candidate on trees)."""
    ind = _indptr(q_indptr)
    if max_path is None:
        max_path = path.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sd_sample_accept(len(ind) - 1, ind, int(vocab), float(temperature), _ptr(logits), _ptr(draft_probs),
                                   _ptr(parents), _ptr(draft_tokens), _ptr(r_accept), _ptr(r_sample),
                                   _ptr(accept_len), _ptr(path), _ptr(out_tokens), int(max_path), _ptr(workspace),
                                   ws_bytes, _ptr(dev_status), _stream(stream)),
           "sd_sample_accept")


def _ptr_array(ts) -> ctypes.Array:
    return (ctypes.c_void_p * len(ts))(*[_ptr(t) for t in ts])


def sd_kv_commit(shape: Shape, k_cache_layers, v_cache_layers, k_new_layers, v_new_layers, page_table,
                 ctx_lens, new_ctx_lens, accept_len, path, max_path: int | None = None, dev_status=None,
                 stream=None) -> None:
    n = len(k_cache_layers)
    if not (len(v_cache_layers) == len(k_new_layers) == len(v_new_layers) == n):
        raise ValueError("per-layer pointer lists differ in length")
    if max_path is None:
        max_path = path.shape[-1]
    _check(load().sd_kv_commit(shape.ref, n, _ptr_array(k_cache_layers), _ptr_array(v_cache_layers),
                               _ptr_array(k_new_layers), _ptr_array(v_new_layers), _ptr(page_table),
                               _ptr(ctx_lens), _ptr(new_ctx_lens), _ptr(accept_len), _ptr(path),
                               int(max_path), _ptr(dev_status), _stream(stream)),
           "sd_kv_commit")


def sd_kv_commit_fp8(shape: Shape, k_cache_layers, v_cache_layers, k_scales, v_scales, k_new_layers,
                     v_new_layers, page_table, ctx_lens, new_ctx_lens, accept_len, path,
                     max_path: int | None = None, dev_status=None, stream=None) -> None:
    """sd_kv_commit into e4m3 caches: the accepted rows are quantised with the per-layer scales."""
    n = len(k_cache_layers)
    if not (len(v_cache_layers) == len(k_new_layers) == len(v_new_layers) == len(k_scales) == len(v_scales) == n):
        raise ValueError("per-layer lists differ in length")
    if max_path is None:
        max_path = path.shape[-1]
    ks = (ctypes.c_float * n)(*[float(x) for x in k_scales])
    vs = (ctypes.c_float * n)(*[float(x) for x in v_scales])
    _check(load().sd_kv_commit_fp8(shape.ref, n, _ptr_array(k_cache_layers), _ptr_array(v_cache_layers), ks, vs,
                                   _ptr_array(k_new_layers), _ptr_array(v_new_layers), _ptr(page_table),
                                   _ptr(ctx_lens), _ptr(new_ctx_lens), _ptr(accept_len), _ptr(path),
                                   int(max_path), _ptr(dev_status), _stream(stream)),
           "sd_kv_commit_fp8")


def sd_ddtree_workspace_size(batch: int, positions: int, vocab: int, topk: int) -> int:
    return int(load().sd_ddtree_workspace_size(int(batch), int(positions), int(vocab), int(topk)))


def sd_ddtree_build(draft_logits, topk: int, budget: int, root_tokens, parents, tokens, scores=None,
                    workspace=None, dev_status=None, stream=None) -> None:
    """draft_logits fp32 [batch, positions, vocab]; parents/tokens int32 [batch, 1 + budget]."""
    batch, positions, vocab = (int(x) for x in draft_logits.shape)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sd_ddtree_build(batch, positions, vocab, int(topk), int(budget), _ptr(draft_logits),
                                  _ptr(root_tokens), _ptr(parents), _ptr(tokens), _ptr(scores), _ptr(workspace),
                                  ws_bytes, _ptr(dev_status), _stream(stream)),
           "sd_ddtree_build")


class GdnShape:
    """An sd_gdn_shape with its host q_indptr kept alive (head_dim 128)."""

    def __init__(self, q_indptr, num_k_heads: int, num_v_heads: int, head_dim: int = 128):
        self.indptr = _indptr(q_indptr)
        self.c = SdGdnShape(len(self.indptr) - 1, ctypes.cast(self.indptr, ctypes.POINTER(ctypes.c_int)),
                            int(num_k_heads), int(num_v_heads), int(head_dim))

    @property
    def ref(self):
        return ctypes.byref(self.c)


def sd_gdn_tree_cache_size(shape: GdnShape) -> int:
    return int(load().sd_gdn_tree_cache_size(shape.ref))


def sd_gdn_conv_tree(q_indptr, x, weight, conv_state, parents, y, dev_status=None, stream=None) -> None:
    """x, y bf16 [sumN, C]; weight fp32 [C, 4]; conv_state bf16 [B, C, 3]."""
    ind = _indptr(q_indptr)
    _check(load().sd_gdn_conv_tree(len(ind) - 1, ind, int(x.shape[-1]), _ptr(x), _ptr(weight), _ptr(conv_state),
                                   _ptr(parents), _ptr(y), _ptr(dev_status), _stream(stream)),
           "sd_gdn_conv_tree")


def sd_gdn_tree(shape: GdnShape, q, k, v, g, beta, state, parents, out, tree_cache, dev_status=None,
                stream=None) -> None:
    cache_bytes = tree_cache.numel() * tree_cache.element_size()
    _check(load().sd_gdn_tree(shape.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(parents),
                              _ptr(out), _ptr(tree_cache), cache_bytes, _ptr(dev_status), _stream(stream)),
           "sd_gdn_tree")


def sd_gdn_commit(shape: GdnShape, state_layers, tree_cache_layers, accept_len, path, conv_state_layers=None,
                  x_layers=None, max_path: int | None = None, dev_status=None, stream=None) -> None:
    n = len(state_layers)
    if len(tree_cache_layers) != n:
        raise ValueError("per-layer lists differ in length")
    channels = 0
    conv_arr = x_arr = None
    if conv_state_layers is not None:
        if len(conv_state_layers) != n or x_layers is None or len(x_layers) != n:
            raise ValueError("per-layer lists differ in length")
        channels = int(x_layers[0].shape[-1])
        conv_arr, x_arr = _ptr_array(conv_state_layers), _ptr_array(x_layers)
    if max_path is None:
        max_path = path.shape[-1]
    _check(load().sd_gdn_commit(shape.ref, n, _ptr_array(state_layers), _ptr_array(tree_cache_layers), channels,
                                conv_arr, x_arr, _ptr(accept_len), _ptr(path), int(max_path), _ptr(dev_status),
                                _stream(stream)),
           "sd_gdn_commit")
