"""One verify step on the GPU: every layer's attention, then accept, then commit.

The three C-ABI calls run in order on one CUDA stream with no host
synchronisation between them, so a step can also be captured into a CUDA
graph (``VerifyStep.capture``).  This module owns the output buffers and the
workspaces; the inputs (queries, draft K/V, caches, logits, tree, page
table) belong to the caller.
"""
from __future__ import annotations

import numpy as np
import torch

from . import native


class VerifyStep:
    """Buffers and calls for one verify step of a fixed batch shape."""

    def __init__(self, q_indptr, max_pages_per_seq: int, num_pool_pages: int, num_layers: int, vocab: int,
                 device="cuda", num_splits: int = 0, max_path: int | None = None, want_lse: bool = False,
                 window: int = 0, k_scales=None, v_scales=None):
        """``k_scales`` / ``v_scales`` (per-layer floats) select e4m3 caches: attention reads the codes with
        these scales and the commit quantises the accepted rows with them."""
        self.q_indptr = np.asarray(q_indptr, dtype=np.int32)
        self.batch = len(self.q_indptr) - 1
        self.total = int(self.q_indptr[-1])
        self.num_layers = int(num_layers)
        self.vocab = int(vocab)
        self.device = torch.device(device)
        self.shape = native.Shape(self.q_indptr, max_pages_per_seq, num_pool_pages, num_splits, window)
        # layers after the first follow the previous layer's attention, which writes no context state
        self.shape_next = self.shape.with_ctx_stable(True)
        self.fp8 = k_scales is not None
        if self.fp8 and (v_scales is None or len(k_scales) != self.num_layers or len(v_scales) != self.num_layers):
            raise ValueError("e4m3 caches need one K and one V scale per layer")
        self.k_scales = None if k_scales is None else [float(x) for x in k_scales]
        self.v_scales = None if v_scales is None else [float(x) for x in v_scales]
        self.max_path = int(max_path or int(np.diff(self.q_indptr).max()))
        dev = self.device
        ws = native.sd_verify_attn_workspace_size(self.shape)
        self.attn_ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.acc_ws = torch.empty(max(native.sd_accept_workspace_size(self.q_indptr, self.vocab), 1),
                                  dtype=torch.uint8, device=dev)
        self.out = [torch.empty((self.total, 24, 256), dtype=torch.bfloat16, device=dev)
                    for _ in range(self.num_layers)]
        self.lse = ([torch.empty((self.total, 24), dtype=torch.float32, device=dev)
                     for _ in range(self.num_layers)] if want_lse else None)
        self.accept_len = torch.empty(self.batch, dtype=torch.int32, device=dev)
        self.path = torch.empty((self.batch, self.max_path), dtype=torch.int32, device=dev)
        self.out_tokens = torch.empty((self.batch, self.max_path), dtype=torch.int32, device=dev)
        self.target_tokens = torch.empty(self.total, dtype=torch.int32, device=dev)
        self.new_ctx_lens = torch.empty(self.batch, dtype=torch.int32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def attention(self, layer, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, stream=None,
                  ctx_stable: bool = False):
        """One layer's attention.  ``ctx_stable``: the previous kernel on the stream writes no context state
        (sd_shape.ctx_stable), so the context loads may start before it finishes."""
        lse = None if self.lse is None else self.lse[layer]
        shape = self.shape_next if ctx_stable else self.shape
        if self.fp8:
            native.sd_verify_attn_fp8(shape, q, k_cache, v_cache, self.k_scales[layer], self.v_scales[layer],
                                      k_new, v_new, page_table, ctx_lens, parents, self.out[layer], lse,
                                      self.attn_ws, self.dev_status, stream)
        else:
            native.sd_verify_attn(shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents,
                                  self.out[layer], lse, self.attn_ws, self.dev_status, stream)

    def accept(self, logits, parents, draft_tokens, stream=None):
        native.sd_accept(self.q_indptr, self.vocab, logits, parents, draft_tokens, self.accept_len, self.path,
                         self.out_tokens, self.target_tokens, self.max_path, self.acc_ws, self.dev_status,
                         stream)

    def commit(self, k_caches, v_caches, k_news, v_news, page_table, ctx_lens, stream=None):
        if self.fp8:
            native.sd_kv_commit_fp8(self.shape, k_caches, v_caches, self.k_scales, self.v_scales, k_news, v_news,
                                    page_table, ctx_lens, self.new_ctx_lens, self.accept_len, self.path,
                                    self.max_path, self.dev_status, stream)
            return
        native.sd_kv_commit(self.shape, k_caches, v_caches, k_news, v_news, page_table, ctx_lens,
                            self.new_ctx_lens, self.accept_len, self.path, self.max_path, self.dev_status,
                            stream)

    def run(self, q, k_caches, v_caches, k_news, v_news, page_table, ctx_lens, parents, draft_tokens, logits,
            stream=None, commit: bool = True):
        """q/k_caches/v_caches/k_news/v_news are per-layer lists of device tensors."""
        for layer in range(self.num_layers):
            self.attention(layer, q[layer], k_caches[layer], v_caches[layer], k_news[layer], v_news[layer],
                           page_table, ctx_lens, parents, stream, ctx_stable=layer > 0)
        self.accept(logits, parents, draft_tokens, stream)
        if commit:
            self.commit(k_caches, v_caches, k_news, v_news, page_table, ctx_lens, stream)

    def launches_per_step(self, commit: bool = True) -> int:
        """Kernel launches one ``run`` issues (attention split (+ merge), argmax, accept, commit)."""
        merge = 1 if native.sd_verify_attn_workspace_size(self.shape) > 0 else 0
        return self.num_layers * (1 + merge) + 2 + (1 if commit else 0)

    def capture(self, *args, **kwargs) -> torch.cuda.CUDAGraph:
        """Capture ``run(*args, **kwargs)`` into a CUDA graph (inputs must stay at the same addresses)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.run(*args, stream=s, **kwargs)
        torch.cuda.current_stream(self.device).wait_stream(s)
        return g


def device_inputs(w, device="cuda"):
    """Move a synthetic workload's small host arrays to the device (int32)."""
    dev = torch.device(device)
    as_t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)
    return dict(page_table=as_t(w.page_table), ctx_lens=as_t(w.ctx_lens), parents=as_t(w.parents),
                draft_tokens=as_t(w.draft_tokens))
