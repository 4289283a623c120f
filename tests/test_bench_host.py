"""Host-side logic of bench.py that its JSON line rests on, checked without a GPU.

- The algorithmic K/V bytes of a layer reproduce the per-step figures of the
  workload table (4096 B per context token per layer for bf16 caches, 2048 B
  for e4m3, only the W - 1 most recent tokens under a window of W).
- A recorded DRAM-traffic figure is reported only while the sources of the
  kernel it was captured on are unchanged, and is matched per workload.
"""
import os

import pytest

import bench
from speculative_decoding_verify_decode_gb300 import synth


def _kv_bytes_per_step(name):
    w = synth.make_workload(name, device="cpu", layers=1, logits=False)
    n = w.total_nodes
    pages = sum((min(int(L), w.window - 1 if w.window else int(L)) + 15) // 16 for L in w.ctx_lens)
    rest = n * 24 * 512 * 2 + n * 4 * 512 * 2 + pages * 4     # Q/O, draft K/V, page-table entries
    return 16 * (bench.attn_bytes_per_layer(w) - rest), w


@pytest.mark.parametrize("name,table_bytes", [
    ("chain8_ctx4k", 268e6),          # 16 layers x 4096 tokens x 4 KB
    ("ddtree22_ctx32k", 2.147e9),
    ("ddtree22_ctx128k", 8.59e9),
])
def test_kv_bytes_match_the_workload_table(name, table_bytes):
    kv, _ = _kv_bytes_per_step(name)
    assert abs(kv - table_bytes) / table_bytes < 0.005, kv


def test_e4m3_cache_halves_the_kv_bytes():
    kv16, _ = _kv_bytes_per_step("ddtree22_ctx32k")
    kv8, w = _kv_bytes_per_step("ddtree22_ctx32k_fp8")
    assert w.kv == "fp8" and kv8 * 2 == kv16


def test_window_counts_only_the_visible_tokens():
    _, w = _kv_bytes_per_step("chain8_ctx32k_win2048")
    full = synth.make_workload("chain8_ctx32k_win2048", device="cpu", layers=1, logits=False)
    full.window = 0
    visible = bench.attn_bytes_per_layer(w)
    assert w.window == 2048
    # 2047 visible tokens of 4096 B each, against the whole context without the window
    assert bench.attn_bytes_per_layer(full) - visible == (int(w.ctx_lens[0]) - 2047) * 4096 + \
        ((int(w.ctx_lens[0]) + 15) // 16 - (2047 + 15) // 16) * 4


def _write(path, text):
    with open(path, "w") as f:
        f.write(text)


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cuh"
    _write(src, "// version 1\n")
    monkeypatch.setitem(bench.ATTN_SRCS, "attn_ring_kernel", [str(src)])
    sha = bench.kernel_sha("attn_ring_kernel")
    table = tmp_path / "traffic.txt"
    _write(table, "# comment line\n"
                  f"wl_a {sha} 1000 990 10 5.00 attn_ring_kernel<144,0>\n"
                  f"wl_b 000000000000 2000 1990 10 5.00 attn_ring_kernel<144,0>\n"
                  f"wl_c {sha} 3000 2990 10 5.00 some_other_kernel<1>\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(table))
    assert bench.traffic_for("wl_a") == 1000.0
    assert bench.traffic_for("wl_b") is None          # captured on other sources
    assert bench.traffic_for("wl_c") is None          # a kernel whose sources are not tracked
    assert bench.traffic_for("wl_missing") is None
    _write(src, "// version 2\n")                    # the kernel changed after the capture
    assert bench.kernel_sha("attn_ring_kernel") != sha
    assert bench.traffic_for("wl_a") is None


def test_committed_traffic_file_names_tracked_kernels():
    with open(bench.TRAFFIC_FILE) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert lines, "no traffic lines"
    for parts in lines:
        kernel = parts[-1].split("<")[0]
        assert kernel in bench.ATTN_SRCS, parts
        assert len(parts[1]) == 12 and int(parts[2]) == int(parts[3]) + int(parts[4]), parts
        assert all(os.path.exists(p) for p in bench.ATTN_SRCS[kernel])
