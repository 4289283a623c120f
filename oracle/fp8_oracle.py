"""Oracle for the quantised (FP8 e4m3) KV cache: the format, quantise-on-commit
and attention over a quantised cache.

TEST INFRASTRUCTURE ONLY.  Plain, slow CPU reference; only the tests, the smoke
check and the bench's CPU-baseline leg may import it.  It shares no code with
the CUDA path and imports nothing from the product package.

Source: «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (S5),
[24 GB 显存上的 128K 上下文]: the KV cache is stored quantised (Q4_0 there),
quantised once on write, and read quantised by the verify attention.

Readings (each is also listed in the design notes):

* format: e4m3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
  infinities; exponent 15 with mantissa 7 is NaN; largest finite 448;
  exponent 0 is subnormal, m * 2^-9);
* one scale per layer and tensor (K, V): stored code = e4m3(x * (1/scale)),
  with x the bf16 value, 1/scale and the product rounded to fp32, and the
  e4m3 rounding to nearest, ties to the even code, finite values beyond 448
  saturating to 448; a cache value reads back as decode(code) * scale;
* only committed context is quantised: the current step's draft K/V (the
  keys of the verify block itself) are attended in bf16.
"""
from __future__ import annotations

import math

import numpy as np

import oracle.verify_oracle as vo

E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of one e4m3 code (NaN for 0x7F / 0xFF)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(x: float) -> int:
    """Round x to the nearest e4m3 value (ties to the even code), saturating finite
    magnitudes above 448 to 448; the sign of zero is kept; NaN -> 0x7F."""
    x = float(x)
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0x00
    a = abs(x)
    if a >= E4M3_MAX:
        return sign | 0x7E
    if a < 2.0 ** -6:                                   # subnormal range: steps of 2^-9
        q = a / 2.0 ** -9
        m = math.floor(q)
        r = q - m
        if r > 0.5 or (r == 0.5 and m % 2 == 1):
            m += 1
        return sign | m                                 # m == 8 is the smallest normal, code 0x08
    e = math.floor(math.log2(a))
    if 2.0 ** e > a:                                    # guard log2 rounding
        e -= 1
    if 2.0 ** (e + 1) <= a:
        e += 1
    q = (a / 2.0 ** e - 1.0) * 8.0                      # mantissa in units of 1/8
    m = math.floor(q)
    r = q - m
    if r > 0.5 or (r == 0.5 and m % 2 == 1):
        m += 1
    if m == 8:                                          # rounded up into the next binade
        m = 0
        e += 1
    code = ((e + 7) << 3) | m
    if code > 0x7E:                                     # only reachable at the top: saturate
        code = 0x7E
    return sign | code


def quantise(x, scale: float) -> np.ndarray:
    """Codes of x (any shape; float values) for one tensor scale: e4m3(fp32(x) * fp32(1/scale))."""
    inv = np.float32(1.0) / np.float32(scale)
    y = np.asarray(x, dtype=np.float32) * inv
    flat = [e4m3_encode(v) for v in y.reshape(-1)]
    return np.asarray(flat, dtype=np.uint8).reshape(y.shape)


_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def dequantise(codes, scale: float) -> np.ndarray:
    """float64 values of a code array: decode(code) * scale."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)] * float(scale)


def kv_commit_fp8(k_caches, v_caches, k_scales, v_scales, k_news, v_news, page_table, ctx_lens, q_indptr,
                  accept_len, paths):
    """sd_kv_commit on e4m3 caches: the accepted nodes' bf16 K/V rows are quantised
    with their layer's scales and written to positions L .. L + A - 1."""
    kq = [quantise(np.asarray(k, dtype=np.float32), s) for k, s in zip(k_news, k_scales)]
    vq = [quantise(np.asarray(v, dtype=np.float32), s) for v, s in zip(v_news, v_scales)]
    return vo.kv_commit(k_caches, v_caches, kq, vq, page_table, ctx_lens, q_indptr, accept_len, paths)


def verify_attention_fp8(q, k_codes, v_codes, k_scale: float, v_scale: float, k_new, v_new, page_table, ctx_lens,
                         q_indptr, parents, samples=None, window=None):
    """Verify attention over e4m3 caches: the context keys and values read back as
    decode(code) * scale; the draft block's own K/V are bf16 (not yet committed)."""
    return vo.verify_attention(q, dequantise(k_codes, k_scale), dequantise(v_codes, v_scale), k_new, v_new,
                               page_table, ctx_lens, q_indptr, parents, samples=samples, window=window)
