"""The seeded input generators (paged_kv_decode_12_gb300.workloads): the same seed gives
the same inputs, and each workload has the shape, sizes and structure it documents.
CPU only (device draws are exercised on CPU tensors)."""
import math

import numpy as np
import torch

from paged_kv_decode_12_gb300 import workloads as wl


def test_workloads_are_seed_deterministic_and_shaped():
    for name in wl.WORKLOADS:
        a, b = wl.make_workload(name, 12), wl.make_workload(name, 12)
        assert np.array_equal(a.seq_lens, b.seq_lens) and a.pool_pages == b.pool_pages
        assert a.seq_lens.min() >= 1 and a.seq_lens.max() <= wl.MAX_CONTEXT
        assert a.pages_per_layer() * a.layers <= a.pool_pages
    assert not np.array_equal(wl.make_workload("b64", 12).seq_lens, wl.make_workload("b64", 13).seq_lens)
    b64 = wl.make_workload("b64")
    assert b64.batch == 64 and list(b64.seq_lens[:6]) == [1, 16, 17, 32, 33, 2048]
    assert b64.key_outlier_frac == 0.01 and 150 < np.median(b64.seq_lens) < 600
    b256 = wl.make_workload("b256")
    assert b256.batch == 256 and np.all(b256.seq_lens == 2048) and b256.pool_pages == 524288
    b8 = wl.make_workload("b8")
    assert b8.batch == 8 and b8.pool_pages == 4096 * 16
    # KV bytes of one b256 step: 256 x 2048 tokens x 16 layers x 2 KiB (BF16), 1088 B (FP8)
    assert b256.kv_bytes_per_step() == 256 * 2048 * 16 * 2048
    assert b256.kv_bytes_per_step("fp8") == 256 * 2048 * 16 * 1088


def test_host_draws_are_seeded_bf16_normals():
    x = wl.bf16_normal_host(np.random.default_rng(3), (4096,))
    y = wl.bf16_normal_host(np.random.default_rng(3), (4096,))
    assert x.dtype == np.uint16 and np.array_equal(x, y)
    v = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(v.mean()) < 0.1 and 0.9 < v.std() < 1.1
    assert np.array_equal(wl.scale_bf16_by_8(x), ((v * 8).view(np.uint32) >> 16).astype(np.uint16))


def test_permutation_block_tables():
    rng = np.random.default_rng(4)
    lens = np.array([1, 16, 17, 100, 2048], dtype=np.int32)
    bt = wl.permutation_block_tables(rng, lens, 200, 128)
    used = []
    for b, L in enumerate(lens):
        n = math.ceil(int(L) / 16)
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, n:] == -1)
        used += bt[b, :n].tolist()
    assert len(used) == len(set(used)) and max(used) < 200
    assert np.array_equal(bt, wl.permutation_block_tables(np.random.default_rng(4), lens, 200, 128))


def test_trace_schedule_is_seeded_and_in_range():
    a, b = wl.trace_schedule(seed=7, steps=100), wl.trace_schedule(seed=7, steps=100)
    assert [(r.rid, r.arrival_step, r.prompt_len, r.max_new) for r in a] == \
           [(r.rid, r.arrival_step, r.prompt_len, r.max_new) for r in b]
    assert all(8 <= r.prompt_len <= 1024 and 16 <= r.max_new <= 1024 and 0 <= r.arrival_step < 100 for r in a)
    assert 30 < len(a) < 100   # Poisson(0.6) per step


def test_device_draws_on_cpu_tensors():
    t1 = wl.fill_bf16_normal_(torch.empty(10000, dtype=torch.bfloat16), 5)
    t2 = wl.fill_bf16_normal_(torch.empty(10000, dtype=torch.bfloat16), 5)
    assert torch.equal(t1, t2) and abs(float(t1.float().mean())) < 0.05
    pages = 64
    codes = torch.empty((pages, 2, 8, 16, 64), dtype=torch.uint8)
    scales = torch.empty((pages, 2, 8, 16), dtype=torch.float32)
    wl.fill_fp8_pages_(codes, scales, 9, key_outlier_frac=0.05)
    c = codes.numpy()
    assert not np.any((c & 0x7F) == 0x7F)                   # no NaN codes
    s = scales.numpy()
    assert s[:, 1].min() >= 0.005 and s[:, 1].max() <= 0.009  # value scales untouched
    outliers = s[:, 0] > 0.009
    assert 0.01 < outliers.mean() < 0.1 and np.all(s[:, 0][outliers] >= 0.04)
