"""Helpers shared by the GPU parity tests (building, host copies, tolerances)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import oracle.fp8_oracle as fp8_oracle
from speculative_decoding_verify_decode_gb300 import build, native, synth
from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        native.load()
        _built = True


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


LSE_TOL = 4e-3


def attn_bound(ref: np.ndarray) -> float:
    """The contract: max |err| <= 2e-2 * max |ref| + 1e-3."""
    return 2e-2 * float(np.abs(ref).max()) + 1e-3


def tight_bound(ref: np.ndarray) -> float:
    """A stricter check than the contract: bf16 output rounding plus bf16 P."""
    return 1e-2 * float(np.abs(ref).max()) + 1e-6


def check_attention(out: torch.Tensor, ref: np.ndarray, lse: torch.Tensor | None = None,
                    ref_lse: np.ndarray | None = None) -> dict:
    got = f64(out)
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max())
    assert err <= attn_bound(ref), (err, attn_bound(ref))
    assert err <= tight_bound(ref), (err, tight_bound(ref))
    out = {"max_err": err, "max_ref": float(np.abs(ref).max())}
    if lse is not None:
        # the kernel normalises by the sum of the bf16-rounded weights it also
        # multiplies V with, so the log-sum-exp carries bf16 rounding: |d lse| <= ln(1 + 2^-8)
        lerr = float(np.abs(f64(lse) - ref_lse).max())
        assert lerr <= LSE_TOL, lerr
        out["lse_err"] = lerr
    return out


def oracle_attention(w, layer: int, samples=None, window: int | None = None):
    win = getattr(w, "window", 0) if window is None else window
    if getattr(w, "kv", "bf16") == "fp8":
        codes = lambda t: t.detach().cpu().numpy()
        return fp8_oracle.verify_attention_fp8(f32(w.q[layer]), codes(w.k_cache[layer]), codes(w.v_cache[layer]),
                                               w.k_scales[layer], w.v_scales[layer], f32(w.k_new[layer]),
                                               f32(w.v_new[layer]), w.page_table, w.ctx_lens, w.q_indptr,
                                               w.parents, samples=samples, window=win or None)
    return oracle.verify_attention(f32(w.q[layer]), f32(w.k_cache[layer]), f32(w.v_cache[layer]),
                                   f32(w.k_new[layer]), f32(w.v_new[layer]), w.page_table, w.ctx_lens,
                                   w.q_indptr, w.parents, samples=samples, window=win or None)


def gpu_attention(w, layer: int, num_splits: int = 0, want_lse: bool = True, window: int | None = None):
    d = device_inputs(w)
    win = getattr(w, "window", 0) if window is None else window
    fp8 = getattr(w, "kv", "bf16") == "fp8"
    st = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, 1, max(w.vocab, 1), num_splits=num_splits,
                    want_lse=want_lse, window=win, k_scales=[w.k_scales[layer]] if fp8 else None,
                    v_scales=[w.v_scales[layer]] if fp8 else None)
    st.attention(0, w.q[layer], w.k_cache[layer], w.v_cache[layer], w.k_new[layer], w.v_new[layer],
                 d["page_table"], d["ctx_lens"], d["parents"])
    torch.cuda.synchronize()
    return st.out[0], (st.lse[0] if want_lse else None), int(st.dev_status.item())


def workload(parents_list, ctx, seed, scale=1.0 / 16, vocab=4096, p=0.7, table="permuted", spare=2,
             layers=1, logits=True, device="cuda", kv="bf16"):
    w = synth.make_structure(len(parents_list), ctx, parents_list, seed, vocab, [p] * len(parents_list),
                             table=table, spare_pages=spare)
    w.kv = kv
    return synth.fill_tensors(w, layers, seed, device=device, qkv_scale=scale, logits=logits)
