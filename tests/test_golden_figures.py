"""The pages' printed figures (tests/golden/page_figures.txt) against the
framework's geometry and byte accounting."""
import os

from paged_kv_decode_12_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")


def _figures():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


def test_kv_growth_worked_example():
    f = _figures()
    b = wl.kv_bytes_per_token(int(f["kv_growth_layers"]), int(f["kv_growth_heads"]),
                              int(f["kv_growth_head_dim"]), int(f["kv_growth_elem_bytes"]))
    assert b == 2_621_440                                  # exactly 2.5 MiB
    assert abs(b / 2**20 - f["kv_growth_mb_approx"]) < 0.05 * f["kv_growth_mb_approx"]


def test_engine_geometry_matches_pages():
    f = _figures()
    assert wl.PAGE_SIZE == f["page_size_tokens"]
    assert wl.MAX_CONTEXT == f["max_context"]
    assert wl.NUM_Q_HEADS * wl.HEAD_DIM == f["hidden"]
    per_token = wl.kv_bytes_per_token(int(f["layers"]))
    assert per_token == 32 * 1024
    # the default pool holds exactly two full contexts
    assert int(f["default_pool_mib"]) * 2**20 // per_token == 2 * wl.MAX_CONTEXT
    # one page of one layer: 16 tokens' K and V for the 8 KV heads
    assert wl.PAGE_BYTES == wl.PAGE_SIZE * wl.kv_bytes_per_token(1)


def test_workload_byte_accounting():
    w = wl.make_workload("b256")
    assert w.kv_bytes_per_step() == 256 * 2048 * 16 * 2048
    t = wl.make_workload("tiny")
    assert t.kv_bytes_per_step() == (17 + 40) * 2048
