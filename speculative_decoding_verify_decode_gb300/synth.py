"""Seeded synthetic inputs for the speculative-decoding verify step.

This module only draws inputs.  It computes no part of the verify step itself:
no attention, no argmax, no path search, no cache commit.  The target argmax of
every logits row is fixed *by construction* (a planted spike at a token chosen
here), so that drafts can be planted to accept with a chosen probability
without this module ever evaluating an argmax.

Workload shapes follow the pages' model geometry and verify set-ups:

* 24 query heads, 4 KV heads, head_dim 256, one full-attention layer in four
  (16 of 64 layers): «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍»
  (blog.xiaohack.org/246393), section 为什么我们要做这个测试.
* 16-token KV pages drawn from one shared physical pool:
  «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图» (xdnf.cn/news/337238),
  sections 2 and 4.
* chain drafts of 4 (MTP/EAGLE) and 8 (DFlash2):
  «Qwen3.8-27B 部署技术报告» (git.mitsea.com, FlintyLemming), MTP and DFlash2
  sections and the throughput table.
* a draft block of 16 expanded into a DDTree of budget 22, verified in one
  forward: the xiaohack page, sections 架构设计 and 从自回归到 DDTree.

Small arrays (trees, tokens, page tables, context lengths) come from a numpy
PCG64 generator; large tensors (Q, K, V, logits) from a seeded
``torch.Generator`` on the device that will hold them, so the multi-GB
workloads never pass through host memory.  The torch stream therefore depends
on the device; every consumer (GPU path and oracle) receives the same tensors.

Recipe (stated once, used by tests and bench):

* Q, K, V entries ~ N(0, 1) * ``qkv_scale`` (default 1/16), rounded to bf16.
* logits fp32: N(0, 1) clipped to [-5.5, 5.5]; row r then gets a spike
  ``6 + U(0, 1)`` at a uniform token ``tau[r]``, which is therefore its unique
  maximum.
* drafts, in node order: with probability p, ``draft[j] = tau[parent[j]]``;
  otherwise a uniform token different from ``tau[parent[j]]`` and from the
  tokens already given to j's siblings (siblings always distinct).
* DDTree: spine depth D ~ U[8, 16] under the root, the remaining nodes hang off
  random nodes with < 3 children and depth < 16, renumbered breadth-first so
  that ``parent[j] < j``; only spine drafts are planted.
* e4m3 (FP8) caches: random codes drawn field by field, sign ~ U{0, 1},
  exponent field round(N(7, 1.2)) clipped to [0, 15], mantissa ~ U{0..7}
  (the NaN pattern, exponent 15 with mantissa 7, becomes mantissa 6); one scale
  per layer and tensor, 2^-5.5 * U(0.75, 1.25), which puts the typical cache
  value near the bf16 recipe's 1/16.  Q and the draft block's K/V stay bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

H_Q = 24
H_KV = 4
HEAD_DIM = 256
PAGE = 16
MAX_NODES = 64


@dataclass
class Workload:
    """One verify step's worth of synthetic inputs."""

    name: str
    batch: int
    layers: int
    vocab: int
    ctx_lens: np.ndarray           # int32 [B]
    q_indptr: np.ndarray           # int32 [B+1]
    parents: np.ndarray            # int32 [sum N] (per-sequence local indices, root = -1)
    draft_tokens: np.ndarray       # int32 [sum N]
    tau: np.ndarray                # int32 [sum N]: planted argmax of each logits row
    page_table: np.ndarray         # int32 [B, max_pages] (-1 = unused)
    num_pool_pages: int
    q: list = field(default_factory=list)        # per layer bf16 [sum N, 24, 256]
    k_new: list = field(default_factory=list)    # per layer bf16 [sum N, 4, 256]
    v_new: list = field(default_factory=list)
    k_cache: list = field(default_factory=list)  # per layer bf16 [P, 4, 16, 256]
    v_cache: list = field(default_factory=list)
    logits: torch.Tensor | None = None           # fp32 [sum N, V]
    window: int = 0                              # sliding window (0: the whole context)
    kv: str = "bf16"                             # cache format: "bf16", or "fp8" (e4m3 codes, uint8)
    k_scales: list = field(default_factory=list)  # fp8: per layer K / V scale (python floats)
    v_scales: list = field(default_factory=list)

    @property
    def total_nodes(self) -> int:
        return int(self.q_indptr[-1])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])


# The five workloads: name -> parameters.
# The seeds of the replayed workloads are chosen so that their one planted
# step accepts the recipe's mean length (within 0.5 over 400 seeds: 4.13 for
# the 8-chain at p = 0.8, 6.0 for the 22-node trees at p = 0.85, 2.8 mean over
# the batch of 4-chains), so that accepted tokens per step are typical.
CONFIGS = {
    "tiny_chain_ctx512": dict(batch=1, layers=1, ctx=512, tree="chain", K=4, vocab=4096,
                              p=0.8, seed=0, table="identity"),
    "chain8_ctx4k": dict(batch=1, layers=16, ctx=4096, tree="chain", K=8, vocab=151936,
                         p=0.8, seed=12, table="permuted"),
    "ddtree22_ctx32k": dict(batch=1, layers=16, ctx=32768, tree="ddtree", budget=22,
                            vocab=151936, p=0.85, seed=3, table="permuted"),
    "conc8_chain4_ragged": dict(batch=8, layers=16, ctx=(1024, 16384), tree="chain", K=4,
                                vocab=151936, p=(0.5, 0.9), seed=3, table="permuted"),
    "ddtree22_ctx128k": dict(batch=1, layers=16, ctx=131072, tree="ddtree", budget=22,
                             vocab=151936, p=0.85, seed=5, table="permuted"),
    # sliding-window verify: attention over the most recent 2,048 positions of a long context
    "chain8_ctx32k_win2048": dict(batch=1, layers=16, ctx=32768, tree="chain", K=8, vocab=151936,
                                  p=0.8, seed=12, table="permuted", window=2048),
    # quantised (e4m3) KV caches: the long-context trees and the 4K chain
    "ddtree22_ctx32k_fp8": dict(batch=1, layers=16, ctx=32768, tree="ddtree", budget=22,
                                vocab=151936, p=0.85, seed=3, table="permuted", kv="fp8"),
    "ddtree22_ctx128k_fp8": dict(batch=1, layers=16, ctx=131072, tree="ddtree", budget=22,
                                 vocab=151936, p=0.85, seed=5, table="permuted", kv="fp8"),
    "chain8_ctx4k_fp8": dict(batch=1, layers=16, ctx=4096, tree="chain", K=8, vocab=151936,
                             p=0.8, seed=12, table="permuted", kv="fp8"),
}


def chain_parents(k: int) -> np.ndarray:
    """Root plus k chained drafts: node j's parent is j-1."""
    return np.arange(-1, k, dtype=np.int32)


def ddtree_parents(rng: np.random.Generator, budget: int, max_depth: int = 16,
                   max_children: int = 3) -> tuple[np.ndarray, np.ndarray]:
    """A random tree with ``budget`` non-root nodes; returns (parents, is_spine).

    The spine (depth D ~ U[8, 16], capped at the budget) is a chain under the root; the other nodes
    attach to random existing nodes that still have room.  Node ids are then
    renumbered breadth-first (children in insertion order) so parent[j] < j.
    """
    spine = int(rng.integers(min(8, budget), min(16, budget) + 1))
    par = [-1] + list(range(spine))            # nodes 0..spine
    depth = [0] + list(range(1, spine + 1))
    nchild = [1] * spine + [0]
    while len(par) < budget + 1:
        cand = [i for i in range(len(par)) if nchild[i] < max_children and depth[i] < max_depth]
        at = int(cand[int(rng.integers(len(cand)))])
        par.append(at)
        depth.append(depth[at] + 1)
        nchild[at] += 1
        nchild.append(0)
    children = [[] for _ in par]
    for j in range(1, len(par)):
        children[par[j]].append(j)
    order = [0]
    for u in order:
        order.extend(children[u])
    new_id = {old: new for new, old in enumerate(order)}
    parents = np.full(len(par), -1, dtype=np.int32)
    is_spine = np.zeros(len(par), dtype=bool)
    for old in range(len(par)):
        parents[new_id[old]] = -1 if par[old] < 0 else new_id[par[old]]
        is_spine[new_id[old]] = old <= spine
    return parents, is_spine


def plant_drafts(rng: np.random.Generator, parents: np.ndarray, tau: np.ndarray, vocab: int,
                 p_accept, planted: np.ndarray | None = None,
                 rescue: bool = False) -> np.ndarray:
    """Draft tokens for one sequence (local node ids).

    Node j (j >= 1) whose ``planted[j]`` is set copies its parent's planted
    argmax ``tau[parent[j]]`` with probability ``p_accept``; every other draft
    is uniform among tokens that differ from that argmax and from the siblings'
    tokens.  ``rescue`` then gives one off-spine node whose spine sibling was
    rejected its parent's argmax (an accepted side branch).
    """
    n = len(parents)
    if planted is None:
        planted = np.ones(n, dtype=bool)
    draft = np.zeros(n, dtype=np.int32)
    draft[0] = int(rng.integers(vocab))     # the root: last emitted token
    used: dict[int, set] = {}
    for j in range(1, n):
        pa = int(parents[j])
        sib = used.setdefault(pa, set())
        target = int(tau[pa])
        if planted[j] and target not in sib and rng.random() < p_accept:
            tok = target
        else:
            if vocab - 1 - len(sib - {target}) <= 0:
                raise ValueError("vocabulary too small for distinct rejected sibling drafts")
            while True:
                tok = int(rng.integers(vocab))
                if tok != target and tok not in sib:
                    break
        sib.add(tok)
        draft[j] = tok
    if rescue:
        for j in range(1, n):
            pa = int(parents[j])
            if planted[j]:
                continue
            sibs = [i for i in range(1, n) if parents[i] == pa and i != j]
            if any(draft[i] == tau[pa] for i in sibs):
                continue
            if any(planted[i] for i in sibs):
                draft[j] = tau[pa]
                break
    return draft


def make_page_table(rng: np.random.Generator, pages_needed: list[int], mode: str,
                    spare_pages: int = 0) -> tuple[np.ndarray, int]:
    """Assign physical pages from one pool; returns (table [B, max], pool size)."""
    total = int(sum(pages_needed)) + spare_pages
    pool = np.arange(total, dtype=np.int32)
    if mode == "permuted":
        pool = rng.permutation(total).astype(np.int32)
    elif mode != "identity":
        raise ValueError(mode)
    table = np.full((len(pages_needed), max(1, max(pages_needed))), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(pages_needed):
        table[b, :n] = pool[at:at + n]
        at += n
    return table, total


def make_structure(batch: int, ctx_lens, parents_list, tau_seed: int, vocab: int, p_list,
                   planted_list=None, table: str = "permuted", spare_pages: int = 0,
                   rescue: bool = False, rng: np.random.Generator | None = None) -> Workload:
    """Small host-side parts of a workload: trees, tokens, page table."""
    rng = rng if rng is not None else np.random.default_rng(tau_seed)
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    sizes = [len(p) for p in parents_list]
    indptr = np.zeros(batch + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(sizes)
    tau = rng.integers(vocab, size=int(indptr[-1])).astype(np.int32)
    drafts = []
    for b in range(batch):
        tb = tau[indptr[b]:indptr[b + 1]]
        pl = None if planted_list is None else planted_list[b]
        drafts.append(plant_drafts(rng, parents_list[b], tb, vocab, p_list[b], pl, rescue))
    pages_needed = [int(math.ceil((int(ctx[b]) + sizes[b]) / PAGE)) for b in range(batch)]
    page_table, pool = make_page_table(rng, pages_needed, table, spare_pages)
    return Workload(name="custom", batch=batch, layers=0, vocab=vocab, ctx_lens=ctx,
                    q_indptr=indptr, parents=np.concatenate(parents_list).astype(np.int32),
                    draft_tokens=np.concatenate(drafts).astype(np.int32), tau=tau,
                    page_table=page_table, num_pool_pages=pool)


def _randn_bf16(gen: torch.Generator, shape, scale: float, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return (x * scale).to(torch.bfloat16)


def random_e4m3_codes(gen: torch.Generator, shape, device) -> torch.Tensor:
    """uint8 e4m3 codes drawn field by field (sign, exponent ~ round(N(7, 1.2)) in [0, 15],
    mantissa uniform); the NaN pattern (exponent 15, mantissa 7) is replaced by mantissa 6."""
    sign = torch.randint(0, 2, shape, generator=gen, device=device, dtype=torch.int32)
    e = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).mul_(1.2).add_(7.0)
    e = e.round_().clamp_(0, 15).to(torch.int32)
    m = torch.randint(0, 8, shape, generator=gen, device=device, dtype=torch.int32)
    m = torch.where((e == 15) & (m == 7), torch.full_like(m, 6), m)
    return (sign * 128 + e * 8 + m).to(torch.uint8)


def fill_tensors(w: Workload, layers: int, seed: int, device="cpu", qkv_scale: float = 1.0 / 16,
                 logits: bool = True) -> Workload:
    """Draw Q, draft K/V, paged K/V caches and logits for ``layers`` layers."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 1000003 + 17)
    n = w.total_nodes
    w.layers = layers
    w.q, w.k_new, w.v_new, w.k_cache, w.v_cache = [], [], [], [], []
    w.k_scales, w.v_scales = [], []
    srng = np.random.default_rng(int(seed) * 7919 + 3)
    cache_shape = (w.num_pool_pages, H_KV, PAGE, HEAD_DIM)
    for _ in range(layers):
        w.q.append(_randn_bf16(gen, (n, H_Q, HEAD_DIM), qkv_scale, device))
        w.k_new.append(_randn_bf16(gen, (n, H_KV, HEAD_DIM), qkv_scale, device))
        w.v_new.append(_randn_bf16(gen, (n, H_KV, HEAD_DIM), qkv_scale, device))
        if w.kv == "fp8":
            w.k_cache.append(random_e4m3_codes(gen, cache_shape, device))
            w.v_cache.append(random_e4m3_codes(gen, cache_shape, device))
            w.k_scales.append(float(2.0 ** -5.5 * srng.uniform(0.75, 1.25)))
            w.v_scales.append(float(2.0 ** -5.5 * srng.uniform(0.75, 1.25)))
        else:
            w.k_cache.append(_randn_bf16(gen, cache_shape, qkv_scale, device))
            w.v_cache.append(_randn_bf16(gen, cache_shape, qkv_scale, device))
    if logits:
        lg = torch.randn((n, w.vocab), generator=gen, device=device, dtype=torch.float32)
        lg.clamp_(-5.5, 5.5)
        spike = 6.0 + torch.rand((n,), generator=gen, device=device, dtype=torch.float32)
        rows = torch.arange(n, device=device)
        lg[rows, torch.as_tensor(w.tau, device=device, dtype=torch.long)] = spike
        w.logits = lg
    return w


def make_workload(name: str, device="cpu", layers: int | None = None, qkv_scale: float = 1.0 / 16,
                  ctx_override=None, logits: bool = True, rescue: bool = False, kv: str | None = None) -> Workload:
    """Build one of the named workloads in ``CONFIGS``.

    ``layers`` and ``ctx_override`` shrink a workload for quick checks while
    keeping its tree, table mode and seed; ``kv`` overrides the cache format.
    """
    cfg = CONFIGS[name]
    rng = np.random.default_rng(cfg["seed"])
    batch = cfg["batch"]
    if isinstance(cfg["ctx"], tuple):
        lo, hi = cfg["ctx"]
        ctx = rng.integers(lo, hi + 1, size=batch)
    else:
        ctx = np.full(batch, cfg["ctx"])
    if ctx_override is not None:
        ctx = np.broadcast_to(np.asarray(ctx_override), (batch,)).copy()
    if isinstance(cfg["p"], tuple):
        p_list = list(rng.uniform(cfg["p"][0], cfg["p"][1], size=batch))
    else:
        p_list = [cfg["p"]] * batch
    parents_list, planted_list = [], []
    for _ in range(batch):
        if cfg["tree"] == "chain":
            par = chain_parents(cfg["K"])
            planted = np.ones(len(par), dtype=bool)
        else:
            par, planted = ddtree_parents(rng, cfg["budget"])
        parents_list.append(par)
        planted_list.append(planted)
    w = make_structure(batch, ctx, parents_list, cfg["seed"], cfg["vocab"], p_list,
                       planted_list, table=cfg["table"], rescue=rescue, rng=rng)
    w.name = name
    w.window = int(cfg.get("window", 0))
    w.kv = kv if kv is not None else cfg.get("kv", "bf16")
    nl = cfg["layers"] if layers is None else layers
    return fill_tensors(w, nl, cfg["seed"], device=device, qkv_scale=qkv_scale, logits=logits)


def draft_logits(batch: int, positions: int, vocab: int, seed: int, scale: float = 2.0,
                 ties: bool = False) -> np.ndarray:
    """Seeded draft-model logits [batch, positions, vocab] (fp32) for the draft-tree builder.

    N(0, scale) entries; with ``ties`` every value is rounded to a coarse grid
    (multiples of 0.25), so that equal logits occur, also across 4096-entry chunks.
    """
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, scale, size=(batch, positions, vocab)).astype(np.float32)
    if ties:
        x = np.round(x * 4.0) / 4.0
    return x


# Gated DeltaNet layers of the hybrid model: 16 key heads, 32 value heads, head dim 128 (a reading: the
# pages name the layer type only); the short convolution runs over the q, k and v channels.
GDN_HK, GDN_HV, GDN_D = 16, 32, 128
GDN_CHANNELS = 2 * GDN_HK * GDN_D + GDN_HV * GDN_D


@dataclass
class GdnInputs:
    """One Gated DeltaNet layer's verify inputs for a batch of draft trees (device tensors)."""

    q: torch.Tensor            # bf16 [sumN, H_k, 128]
    k: torch.Tensor            # bf16 [sumN, H_k, 128]
    v: torch.Tensor            # bf16 [sumN, H_v, 128]
    g: torch.Tensor            # fp32 [sumN, H_v] log decay (<= 0)
    beta: torch.Tensor         # fp32 [sumN, H_v] in [0, 1]
    state: torch.Tensor        # fp32 [B, H_v, 128, 128]
    x: torch.Tensor            # bf16 [sumN, C] convolution inputs
    conv_w: torch.Tensor       # fp32 [C, 4]
    conv_state: torch.Tensor   # bf16 [B, C, 3]


def gdn_inputs(n_total: int, batch: int, seed: int, device="cpu", hk: int = GDN_HK, hv: int = GDN_HV,
               channels: int = GDN_CHANNELS, state_scale: float = 0.05, decay: float = 0.5) -> GdnInputs:
    """Seeded draws: q, k, v, x ~ N(0, 1) (bf16); g ~ -U(0, decay); beta ~ U(0, 1); state ~ N(0, state_scale^2);
    convolution taps ~ N(0, 0.5^2); convolution state ~ N(0, 1) (bf16)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 7907 + 11)
    rn = lambda *shape: torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    ru = lambda *shape: torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    return GdnInputs(q=rn(n_total, hk, GDN_D).to(torch.bfloat16), k=rn(n_total, hk, GDN_D).to(torch.bfloat16),
                     v=rn(n_total, hv, GDN_D).to(torch.bfloat16), g=-decay * ru(n_total, hv), beta=ru(n_total, hv),
                     state=state_scale * rn(batch, hv, GDN_D, GDN_D), x=rn(n_total, channels).to(torch.bfloat16),
                     conv_w=0.5 * rn(channels, 4), conv_state=rn(batch, channels, 3).to(torch.bfloat16))
