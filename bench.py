"""Benchmark of the speculative-decoding verify step on one GB300 (or N replicas).

A step is one pass of the whole hot path over one synthetic batch: verify
attention for every layer, argmax + greedy accept, and the KV commit of all
layers.  The default workload is the long-context tree verify: a 22-node draft
tree at 131072 tokens of context (16 layers, 24/4 heads, d = 256, bf16 paged KV
with a permuted page table, logits [23, 151936]); ``--config`` picks another
one.  The other four workloads of the set are timed after it, more briefly,
and reported under ``workloads`` (``--no-extra`` skips them).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
baseline arm), on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verify_decode_gb300 import native, synth  # noqa: E402
from speculative_decoding_verify_decode_gb300.step import VerifyStep, device_inputs  # noqa: E402

METRIC = "verify steps/s"
DEFAULT_CONFIG = "ddtree22_ctx128k"
EXTRA_CONFIGS = ["tiny_chain_ctx512", "chain8_ctx4k", "ddtree22_ctx32k", "conc8_chain4_ragged"]
CSRC = os.path.join(ROOT, "speculative_decoding_verify_decode_gb300", "csrc")
# the sources of each attention kernel: a traffic figure holds while they are unchanged
ATTN_SRCS = {"attn_ring_kernel": [os.path.join(CSRC, f) for f in ("attn_ring_kernel.cuh", "attn_ring_launch.cuh",
                                                                  "attn_ring.cu", "attn_ring_win.cu", "tc_ptx.cuh")],
             "attn_tc_kernel": [os.path.join(CSRC, f) for f in ("attn_tc_kernel.cuh", "attn_tc8.cu", "attn_tc16.cu",
                                                                "tc_ptx.cuh")]}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_traffic.txt")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def attn_bytes_per_layer(w) -> int:
    """Algorithmic bytes of one layer's verify attention.

    Context K and V are read once (2 x 4 heads x 256 x 2 B = 4096 B per token;
    2048 B with e4m3 caches), plus Q, the draft K/V, the output and the
    page-table entries.  With a sliding window W only the W - 1 most recent
    context tokens are visible.
    """
    lens = [int(L) for L in w.ctx_lens]
    if getattr(w, "window", 0):
        lens = [min(L, w.window - 1) for L in lens]
    ctx = sum(lens)
    pages = int(sum((L + 15) // 16 for L in lens))
    n = w.total_nodes
    per_token = 2048 if getattr(w, "kv", "bf16") == "fp8" else 4096
    return ctx * per_token + n * 24 * 512 * 2 + n * 4 * 512 * 2 + pages * 4


def kernel_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for src in ATTN_SRCS[kernel]:
        with open(src, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def traffic_for(config: str):
    """dram bytes per attention launch from the last ncu capture of the workload, if the captured kernel's
    sources (the kernel name ends each line) are unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == config:
                    kernel = parts[-1].split("<")[0]
                    return float(parts[2]) if kernel in ATTN_SRCS and parts[1] == kernel_sha(kernel) else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- GPU arm

def time_ddtree_build(dev, stream, batch: int, budget: int, positions: int = 16, vocab: int = 151936,
                      topk: int = 8, reps: int = 50) -> dict:
    """The draft-tree construction that precedes a tree verify step, timed on its own: top-8 of
    every draft position's logits, then the best-first tree of `budget` nodes (one draft block of
    16 positions per sequence, as on the DDTree page)."""
    logits = torch.from_numpy(synth.draft_logits(batch, positions, vocab, seed=17)).to(dev)
    roots = torch.zeros(batch, dtype=torch.int32, device=dev)
    par = torch.empty((batch, 1 + budget), dtype=torch.int32, device=dev)
    tok = torch.empty_like(par)
    ws = torch.empty(native.sd_ddtree_workspace_size(batch, positions, vocab, topk), dtype=torch.uint8,
                     device=dev)
    for _ in range(3):
        native.sd_ddtree_build(logits, topk, budget, roots, par, tok, None, ws, stream=stream)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        native.sd_ddtree_build(logits, topk, budget, roots, par, tok, None, ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1000.0 / reps
    gbs = batch * positions * vocab * 4 / (us * 1e-6) / 1e9
    peak, _ = peaks()
    return {"us": us, "logits_gbs": gbs, "frac": gbs / peak, "launches": 2,
            "shape": {"batch": batch, "positions": positions, "vocab": vocab, "topk": topk, "budget": budget}}


GDN_LAYERS = 48    # Gated DeltaNet layers of the hybrid model (48 of 64)


def gdn_bytes_per_layer(batch: int, n_total: int) -> dict:
    """Algorithmic bytes of one Gated DeltaNet layer's tree verify and of its commit.

    Tree rule: the cached state (H_v x 128 x 128 fp32 = 64 KB per value head) is read once per sequence;
    q and k (H_k x 128 bf16), v and o (H_v x 128 bf16), g and beta (fp32) per node; the tree cache it
    writes (u: H_v x 128 fp32, normalised keys: H_k x 128 fp32, log decays).  Convolution: x and y
    (C bf16) per node, the taps (C x 4 fp32) and the convolution state (C x 3 bf16) per sequence.
    Commit: the state is read and written once; the path's cache rows are read.
    """
    hk, hv, d, c = synth.GDN_HK, synth.GDN_HV, synth.GDN_D, synth.GDN_CHANNELS
    state = batch * hv * d * d * 4
    tree = state + n_total * (2 * hk * d * 2 + 2 * hv * d * 2 + hv * 8 + hv * d * 4 + hk * d * 4 + hv * 4)
    conv = n_total * c * 4 + c * 16 + batch * c * 6
    return {"tree": tree, "conv": conv, "commit": 2 * state}


def time_gdn(dev, stream, w, reps: int) -> dict:
    """The hybrid layers' verify for the workload's draft trees: per layer the tree convolution and the tree
    gated delta rule (48 layers in one CUDA graph), then persist-on-accept of all 48 layers in one launch."""
    n, B = w.total_nodes, w.batch
    parents = torch.as_tensor(w.parents, dtype=torch.int32, device=dev)
    shape = native.GdnShape(w.q_indptr, synth.GDN_HK, synth.GDN_HV)
    ins = [synth.gdn_inputs(n, B, 100 + layer, device=dev) for layer in range(GDN_LAYERS)]
    caches = [torch.empty(native.sd_gdn_tree_cache_size(shape), dtype=torch.uint8, device=dev) for _ in ins]
    outs = [torch.empty_like(x.v) for x in ins]
    ys = [torch.empty_like(x.x) for x in ins]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # a valid accept result: every sequence keeps its root only (A = 1)
    lens = torch.ones(B, dtype=torch.int32, device=dev)
    path = torch.zeros((B, 1), dtype=torch.int32, device=dev)

    def layers(s):
        for x, cache, out, y in zip(ins, caches, outs, ys):
            native.sd_gdn_conv_tree(w.q_indptr, x.x, x.conv_w, x.conv_state, parents, y, status, stream=s)
            native.sd_gdn_tree(shape, x.q, x.k, x.v, x.g, x.beta, x.state, parents, out, cache, status, stream=s)

    def commit(s):
        native.sd_gdn_commit(shape, [x.state for x in ins], caches, lens, path,
                             conv_state_layers=[x.conv_state for x in ins], x_layers=[x.x for x in ins],
                             dev_status=status, stream=s)

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                fn(cap)
        stream.wait_stream(cap)
        return g

    g_layers, g_commit = graph_of(layers), graph_of(commit)
    res = {}
    for name, g in (("layers", g_layers), ("commit", g_commit)):
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = e0.elapsed_time(e1) * 1000.0 / reps
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the hybrid layers")
    # the tree rule alone (the dominant kernel of the hybrid layers)
    g_tree = graph_of(lambda s: [native.sd_gdn_tree(shape, x.q, x.k, x.v, x.g, x.beta, x.state, parents, out, cache,
                                                    status, stream=s) for x, cache, out in zip(ins, caches, outs)])
    for _ in range(3):
        g_tree.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g_tree.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    tree_us = e0.elapsed_time(e1) * 1000.0 / (reps * GDN_LAYERS)
    by = gdn_bytes_per_layer(B, n)
    peak, _ = peaks()
    tree_gbs = by["tree"] / (tree_us * 1e-6) / 1e9
    commit_gbs = GDN_LAYERS * by["commit"] / (res["commit"] * 1e-6) / 1e9
    return {"layers": GDN_LAYERS, "heads": f"{synth.GDN_HK}k/{synth.GDN_HV}v", "head_dim": synth.GDN_D,
            "conv_channels": synth.GDN_CHANNELS, "us_per_step_layers": res["layers"],
            "us_per_layer": res["layers"] / GDN_LAYERS, "tree_us_per_layer": tree_us,
            "tree_alg_bytes_per_layer": by["tree"], "tree_gbs": tree_gbs, "tree_frac": tree_gbs / peak,
            "commit_us": res["commit"], "commit_gbs": commit_gbs, "commit_frac": commit_gbs / peak,
            "launches_per_step": 2 * GDN_LAYERS + 2}


def time_sample_accept(dev, stream, w, reps: int, temperature: float = 1.0) -> dict:
    """Sampling-based verify of the workload's draft blocks (in place of the greedy accept): the target logits
    of the step, a draft distribution per node (softmax of the logits plus noise), drafts and uniforms drawn
    once; timed from a CUDA graph."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    n, V = w.total_nodes, w.vocab
    q = torch.softmax((w.logits + 0.5 * torch.randn((n, V), generator=g, device=dev)) / temperature, dim=-1)
    parents = torch.as_tensor(w.parents, dtype=torch.int32, device=dev)
    drafts = torch.as_tensor(w.draft_tokens, dtype=torch.int32, device=dev)
    r_acc = torch.rand(n, generator=g, device=dev)
    r_smp = torch.rand(n, generator=g, device=dev)
    max_path = int(np.diff(w.q_indptr).max())
    ws = torch.empty(native.sd_sample_accept_workspace_size(w.q_indptr, V), dtype=torch.uint8, device=dev)
    lens = torch.empty(w.batch, dtype=torch.int32, device=dev)
    path = torch.empty((w.batch, max_path), dtype=torch.int32, device=dev)
    toks = torch.empty((w.batch, max_path), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call(s):
        native.sd_sample_accept(w.q_indptr, V, temperature, w.logits, q, parents, drafts, r_acc, r_smp, lens, path,
                                toks, max_path, ws, status, stream=s)

    gr = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gr, stream=cap):
            call(cap)
    stream.wait_stream(cap)
    for _ in range(3):
        gr.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        gr.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the sampling verify")
    us = e0.elapsed_time(e1) * 1000.0 / reps
    # algorithmic bytes: the statistics pass reads the logits, the first-residual pass logits and draft rows
    alg = n * V * 12
    peak, _ = peaks()
    return {"us": us, "temperature": temperature, "accepted_tokens": int(lens.sum().item()),
            "alg_bytes": alg, "gbs": alg / (us * 1e-6) / 1e9, "frac": alg / (us * 1e-6) / 1e9 / peak, "launches": 3}


def measure(config: str, dev, stream, steps: int, warmup: int, world: int, splits: int = 0, layers=None,
            clocks_index=None) -> dict:
    """Time one workload: the whole step (a CUDA graph replayed `steps` times between events), every
    layer's verify attention alone (the dominant kernel), and the step end to end with host inputs and
    results.  Returns the numbers and the objects the headline line reuses."""
    w = synth.make_workload(config, device=dev, layers=layers)
    d = device_inputs(w, dev)
    fp8 = w.kv == "fp8"
    step = VerifyStep(w.q_indptr, w.max_pages, w.num_pool_pages, w.layers, w.vocab, device=dev,
                      num_splits=splits, window=w.window, k_scales=w.k_scales if fp8 else None,
                      v_scales=w.v_scales if fp8 else None)
    run_args = (w.q, w.k_cache, w.v_cache, w.k_new, w.v_new, d["page_table"], d["ctx_lens"], d["parents"],
                d["draft_tokens"], w.logits)
    step.run(*run_args)                       # eager once: surfaces launch errors early
    torch.cuda.synchronize(dev)
    graph = step.capture(*run_args)
    for _ in range(max(warmup, 3)):
        graph.replay()
    torch.cuda.synchronize(dev)
    status = int(step.dev_status.item())
    if status != 0:
        raise RuntimeError(f"{config}: device status {status} after warm-up")
    accepted = int(step.accept_len.sum().item())

    # ---- timed region: `steps` steps, graph replays back to back
    barrier(world)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(clocks_index) if clocks_index is not None else None
    if clk is not None:
        clk.__enter__()
    t0.record(stream)
    for _ in range(steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if clk is not None:
        clk.__exit__(None, None, None)
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = ms / steps

    # ---- the dominant kernel: every layer's verify attention captured in one
    # graph, replayed between events on the launching stream
    attn_graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(attn_graph, stream=cap):
            for layer in range(w.layers):
                step.attention(layer, w.q[layer], w.k_cache[layer], w.v_cache[layer], w.k_new[layer],
                               w.v_new[layer], d["page_table"], d["ctx_lens"], d["parents"], stream=cap,
                               ctx_stable=layer > 0)
    stream.wait_stream(cap)
    for _ in range(3):
        attn_graph.replay()
    reps = max(5, steps // 2)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(reps):
        attn_graph.replay()
    a1.record(stream)
    torch.cuda.synchronize(dev)
    attn_ms = a0.elapsed_time(a1) / (reps * w.layers)
    peak, peak_kind = peaks()
    alg = attn_bytes_per_layer(w)
    achieved = alg / (attn_ms * 1e-3) / 1e9

    # ---- end to end through the public API: host inputs in, host results out.  As a serving loop
    # would, the step's inputs (every layer's Q and draft K/V, the logits, the tree and the draft
    # tokens) live in one pinned host buffer and one device buffer (aligned views), so a step moves
    # them with one copy; one CUDA graph holds that copy, the step (VerifyStep.run, as above) and the
    # read of its results.
    in_list = list(w.q) + list(w.k_new) + list(w.v_new) + [w.logits, d["parents"], d["draft_tokens"]]
    out_list = [step.accept_len, step.path, step.out_tokens, step.new_ctx_lens]

    def layout(ts):
        offs, at = [], 0
        for x in ts:
            offs.append(at)
            at += (x.numel() * x.element_size() + 255) // 256 * 256
        return offs, at

    def views(buf, ts, offs):
        return [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o in zip(ts, offs)]

    in_offs, in_bytes = layout(in_list)
    out_offs, out_bytes = layout(out_list)
    dev_in_buf = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    host_in_buf = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    dev_out_buf = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    host_out_buf = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    dev_in = views(dev_in_buf, in_list, in_offs)
    for hv, x in zip(views(host_in_buf, in_list, in_offs), in_list):
        hv.copy_(x.detach().to("cpu"))
    dev_out = views(dev_out_buf, out_list, out_offs)
    L = w.layers
    e2e_args = (dev_in[0:L], w.k_cache, w.v_cache, dev_in[L:2 * L], dev_in[2 * L:3 * L], d["page_table"],
                d["ctx_lens"], dev_in[3 * L + 1], dev_in[3 * L + 2], dev_in[3 * L])
    e2e_graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        dev_in_buf.copy_(host_in_buf, non_blocking=True)
        step.run(*e2e_args, stream=cap)   # warm-up outside the capture
        with torch.cuda.graph(e2e_graph, stream=cap):
            dev_in_buf.copy_(host_in_buf, non_blocking=True)
            step.run(*e2e_args, stream=cap)
            for o, v in zip(out_list, dev_out):
                v.copy_(o)
            host_out_buf.copy_(dev_out_buf, non_blocking=True)
    stream.wait_stream(cap)
    e2e_steps = max(5, steps // 2)
    for _ in range(3):
        e2e_graph.replay()
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    if int(step.dev_status.item()) != 0:
        raise RuntimeError(f"{config}: device status {int(step.dev_status.item())} after the timed runs")
    return {"w": w, "step": step, "fp8": fp8, "ms_per_step": ms_per_step, "accepted": accepted,
            "attn_ms": attn_ms, "alg": alg, "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
            "e2e_ms": e2e_ms, "h2d": in_bytes, "d2h": out_bytes, "clocks": clk.summary() if clk else None}


def config_of(name: str, w, world: int) -> dict:
    """The workload-defining keys of `config`, the same in both arms."""
    per_step = attn_bytes_per_layer(w) * w.layers
    return {"workload": name, "batch": w.batch, "layers": w.layers, "window": w.window, "kv": w.kv,
            "ctx_lens": [int(x) for x in w.ctx_lens][:8], "draft_nodes": w.total_nodes, "vocab": w.vocab,
            "heads": "24q/4kv", "head_dim": 256, "page": 16,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": (f"inputs larger than L2 (KV read per step {per_step / 1e6:.0f} MB > 129 MB)" if per_step > 129e6
                   else f"inputs smaller than L2 (KV read per step {per_step / 1e6:.1f} MB): warm-cache figure")}


def workload_summary(m: dict, world: int) -> dict:
    """The numbers of one workload, as reported under `workloads`."""
    return {"value": world * 1000.0 / m["ms_per_step"], "unit": "steps/s", "ms_per_step": m["ms_per_step"],
            "l2": config_of("", m["w"], world)["l2"],
            "accepted_tok_per_s": world * m["accepted"] * 1000.0 / m["ms_per_step"],
            "attn_us_per_layer": m["attn_ms"] * 1000.0, "kv_read_gbs": m["achieved"],
            "frac": m["achieved"] / m["peak"],
            "e2e": {"value": world * 1000.0 / m["e2e_ms"], "unit": "steps/s", "h2d_bytes_per_step": m["h2d"],
                    "d2h_bytes_per_step": m["d2h"]}}


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    native.load()
    stream = torch.cuda.current_stream(dev)
    m = measure(args.config, dev, stream, args.steps, args.warmup, world, splits=args.splits,
                layers=args.layers or None, clocks_index=local)
    w, step = m["w"], m["step"]
    ms_per_step = m["ms_per_step"]
    line = {
        "metric": METRIC,
        "value": world * 1000.0 / ms_per_step,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 KV, f16 MMA" if m["fp8"] else "bf16",
        "data": ("synthetic (seeded; Q and draft K/V ~ N(0,1)/16 bf16, random e4m3 cache codes with per-layer "
                 "scales, planted-argmax fp32 logits)" if m["fp8"] else
                 "synthetic (seeded; Q/K/V ~ N(0,1)/16 bf16, planted-argmax fp32 logits)"),
        "config": config_of(args.config, w, world),
        "cuda_graph": True,
        "accepted_tokens_per_step": m["accepted"],
        "accepted_tok_per_s": world * m["accepted"] * 1000.0 / ms_per_step,
        "kv_read_gbs": m["achieved"],
        "roofline": {"bound": "hbm", "achieved": m["achieved"], "peak": m["peak"], "unit": "GB/s",
                     "frac": m["achieved"] / m["peak"], "traffic": traffic_for(args.config),
                     "kernel": "verify attention of one layer (split kernel + merge), from a graph of all layers",
                     "alg_bytes_per_launch": m["alg"], "launch_ms": m["attn_ms"], "peak_kind": m["peak_kind"]},
        "e2e": {"value": world * 1000.0 / m["e2e_ms"], "unit": "steps/s", "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": m["d2h"]},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": m["clocks"],
    }
    if args.config.startswith("ddtree"):
        line["ddtree_build"] = time_ddtree_build(dev, stream, w.batch, w.total_nodes // w.batch - 1)
    if not args.no_gdn:
        line["gdn_layers"] = time_gdn(dev, stream, w, reps=max(5, args.steps // 2))
    line["sample_accept"] = time_sample_accept(dev, stream, w, reps=max(5, args.steps // 2))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.config, reps=3)
    del m, w, step
    torch.cuda.empty_cache()
    if not args.no_extra:
        # the other workloads of the set, each timed the same way over fewer steps
        extra = {}
        for cfg in EXTRA_CONFIGS:
            if cfg == args.config:
                continue
            mx = measure(cfg, dev, stream, max(10, args.steps // 2), 3, world, splits=args.splits)
            extra[cfg] = workload_summary(mx, world)
            del mx
            torch.cuda.empty_cache()
        line["workloads"] = extra
    return line


# ---------------------------------------------------------------- CPU oracle arm

def _oracle_sample(w, host, logits):
    """One sample of the oracle: one layer's attention, the accept, one layer's commit (seconds each)."""
    import oracle
    import oracle.fp8_oracle as fp8_oracle
    layer = 0
    fp8 = w.kv == "fp8"
    t = time.perf_counter()
    if fp8:
        fp8_oracle.verify_attention_fp8(host["q"], host["kc"], host["vc"], w.k_scales[layer], w.v_scales[layer],
                                        host["kn"], host["vn"], w.page_table, w.ctx_lens, w.q_indptr,
                                        w.parents, window=w.window or None)
    else:
        oracle.verify_attention(host["q"], host["kc"], host["vc"], host["kn"], host["vn"], w.page_table,
                                w.ctx_lens, w.q_indptr, w.parents, window=w.window or None)
    t_attn = time.perf_counter() - t
    t = time.perf_counter()
    _, lens, paths, _ = oracle.accept(w.q_indptr, w.parents, w.draft_tokens, logits)
    t_acc = time.perf_counter() - t
    t = time.perf_counter()
    if fp8:
        fp8_oracle.kv_commit_fp8([host["kc"]], [host["vc"]], [w.k_scales[layer]], [w.v_scales[layer]],
                                 [host["kn"]], [host["vn"]], w.page_table, w.ctx_lens, w.q_indptr, lens, paths)
    else:
        oracle.kv_commit([host["kc"]], [host["vc"]], [host["kn"]], [host["vn"]], w.page_table, w.ctx_lens,
                         w.q_indptr, lens, paths)
    t_com = time.perf_counter() - t
    return t_attn, t_acc, t_com


def _host_copies(w):
    f32 = lambda x: x.detach().to("cpu", torch.float32).numpy()
    fp8 = w.kv == "fp8"
    cache = (lambda x: x.detach().cpu().numpy()) if fp8 else f32
    host = dict(q=f32(w.q[0]), kc=cache(w.k_cache[0]), vc=cache(w.v_cache[0]), kn=f32(w.k_new[0]),
                vn=f32(w.v_new[0]))
    return host, w.logits.detach().cpu().numpy()


def cpu_baseline(w, config: str, reps: int = 3) -> dict:
    """Time the oracle on a bounded sample: `reps` repetitions of one layer's attention + accept + one
    layer's commit; the median of each part is extrapolated to a step of `w.layers` layers."""
    host, logits = _host_copies(w)
    parts = [_oracle_sample(w, host, logits) for _ in range(reps)]
    t_attn = statistics.median(p[0] for p in parts)
    t_acc = statistics.median(p[1] for p in parts)
    t_com = statistics.median(p[2] for p in parts)
    step_s = w.layers * t_attn + t_acc + w.layers * t_com
    return {"value": 1.0 / step_s, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{config}: median of {reps} x (1 layer attention + accept + 1 layer commit) on the host, "
                      f"extrapolated to {w.layers} layers; numpy fp64",
            "reps": reps, "layers_extrapolated": w.layers,
            "attn_s_per_layer": t_attn, "accept_s": t_acc, "commit_s_per_layer": t_com}


def run_reference(args, world, rank, local):
    """The oracle arm: `warmup` untimed and `steps` timed samples, each one layer's attention + accept + one
    layer's commit.  `ms_per_step` is the measured time of one sample (so steps x ms_per_step is the timed
    wall time); `value` extrapolates the median sample to a whole step of the workload's layers."""
    if rank != 0:
        return None
    w = synth.make_workload(args.config, device="cpu")
    host, logits = _host_copies(w)
    for _ in range(args.warmup):
        _oracle_sample(w, host, logits)
    t = time.perf_counter()
    parts = [_oracle_sample(w, host, logits) for _ in range(max(1, args.steps))]
    wall = time.perf_counter() - t
    t_attn = statistics.median(p[0] for p in parts)
    t_acc = statistics.median(p[1] for p in parts)
    t_com = statistics.median(p[2] for p in parts)
    v = 1.0 / (w.layers * t_attn + t_acc + w.layers * t_com)
    base = {"value": v, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{args.config}: each timed step is 1 layer attention + accept + 1 layer commit on the host "
                      f"(numpy fp64); value extrapolates the median step to {w.layers} layers",
            "reps": len(parts), "layers_extrapolated": w.layers, "wall_s": wall,
            "attn_s_per_layer": t_attn, "accept_s": t_acc, "commit_s_per_layer": t_com}
    return {"metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": world, "steps": len(parts),
            "warmup": args.warmup, "ms_per_step": 1000.0 * wall / len(parts), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": config_of(args.config, w, world),
            "impl": "reference", "timed_step": "1 layer attention + accept + 1 layer commit",
            "layers_extrapolated": w.layers, "cpu_baseline": base,
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gdn", action="store_true", help="skip the hybrid (Gated DeltaNet) layers' timing")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads of the set")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers of the workload to build (0 = its own count; fewer only for profiler captures)")
    ap.add_argument("--splits", type=int, default=0, help="split-KV chunks per (sequence, KV head); 0 = auto")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank, local)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
