"""Pins for the oracle's FP8 KV pages.

The KV-cache tutorial ("从零构建大模型推理引擎：KV缓存、算子融合与量化优化实战",
section 5.1) suggests storing the KV cache in low precision and dequantizing before
attention; the scheme here is a reading: FP8 E4M3 (no infinities, largest 448),
round to nearest even, saturating, one FP32 scale = amax/448 per (token, KV head)
row, code = E4M3(x / scale) with FP32 arithmetic.  Pinned against torch's
float8_e4m3fn conversion (a library routine) in its non-saturating range, closed
forms of the scheme (the row maximum maps to +-448; the dequantization error is at
most half a code step times the scale), and brute-force attention over the
dequantized values laid out contiguously.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_12_gb300 import workloads as wl
from tests import paged_helpers as ph

HQ, HKV, D, PS = wl.NUM_Q_HEADS, wl.NUM_KV_HEADS, wl.HEAD_DIM, wl.PAGE_SIZE
PAGE = oracle.FP8_PAGE_BYTES
CODES = 2 * HKV * PS * D


def torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]) and np.all(np.isnan(got[~ok]))


def test_encode_matches_library_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-448, 448, 4000), rng.standard_normal(4000), rng.uniform(-2.0**-6, 2.0**-6, 2000),
        # exact midpoints between neighbouring codes (ties)
        [(a + b) / 2 for a, b in zip(oracle.e4m3_to_f64(np.arange(0, 126, dtype=np.uint8)),
                                     oracle.e4m3_to_f64(np.arange(1, 127, dtype=np.uint8)))],
    ]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_from_f64(x.astype(np.float64)), torch_e4m3(x))


@pytest.mark.parametrize("value,code", [(448.0, 0x7E), (448.5, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (0.0, 0x00),
                                        (2.0**-9, 0x01), (2.0**-10, 0x00), (3 * 2.0**-10, 0x02), (1.0, 0x38)])
def test_encode_saturation_and_known_codes(value, code):
    assert int(oracle.e4m3_from_f64(np.array([value]))[0]) == code


def test_quantize_row_closed_forms():
    rng = np.random.default_rng(2)
    for _ in range(50):
        row = wl.bf16_normal_host(rng, (D,))
        codes, scale = oracle.quantize_row_fp8(row)
        x = ph.bf16_to_f64(row)
        i = int(np.argmax(np.abs(x)))
        assert codes[i] == (0xFE if x[i] < 0 else 0x7E)                    # the row maximum is +-448
        amax = np.float32(np.abs(x).max())
        assert scale == np.float32(amax / np.float32(448.0))
        # codes = library E4M3 of the FP32 quotient
        assert np.array_equal(codes, torch_e4m3(x.astype(np.float32) / scale))
        xq = oracle.e4m3_to_f64(codes) * float(scale)
        step = np.where(np.abs(x / scale) < 2.0**-6, 2.0**-9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x / scale),
                                                                                         2.0**-6))) - 3))
        assert np.all(np.abs(xq - x) <= 0.5 * step * float(scale) * (1 + 1e-6))
    codes, scale = oracle.quantize_row_fp8(np.zeros(D, dtype=np.uint16))
    assert scale == 1.0 and np.all(codes == 0)


def fp8_pool(num_pages):
    return np.full(num_pages * PAGE, 0xA5, dtype=np.uint8)


UNIT = PAGE // HKV            # one KV head's codes (K rows, interleaved V rows) then scales [2][16]


def test_fp8_decode_equals_contiguous_dequantized():
    rng = np.random.default_rng(3)
    lens = np.array([1, 17, 40, 100], dtype=np.int32)
    num_pages = ph.pages_needed(lens) + 2
    bt = wl.permutation_block_tables(rng, lens, num_pages, 8)
    pool = fp8_pool(num_pages)
    pv = ph.Fp8Pages(pool)
    S = int(lens.max())
    K = np.zeros((len(lens), HKV, S, D))
    V = np.zeros((len(lens), HKV, S, D))
    for b, L in enumerate(lens):
        for t in range(L):
            page, slot = bt[b, t // PS], t % PS
            for kv, dst in ((0, K), (1, V)):
                for h in range(HKV):
                    c, s = oracle.quantize_row_fp8(wl.bf16_normal_host(rng, (D,)))
                    pv.set_row(page, kv, h, slot, c, s)
                    dst[b, h, t] = oracle.e4m3_to_f64(c) * float(s)
    q = wl.bf16_normal_host(rng, (len(lens), HQ, D))
    _, paged = oracle.decode_fp8(pool, oracle.geom(num_pages), bt, lens, q, 1 / 8)
    contiguous = oracle.decode_contiguous(K, V, lens, ph.bf16_to_f64(q), 1 / 8)
    assert np.allclose(paged, contiguous, rtol=0, atol=1e-12)
    # a single token returns its dequantized value
    assert np.allclose(paged[0], V[0, np.arange(HQ) // 4, 0], rtol=0, atol=1e-15)


def test_fp8_append_matches_bf16_append_then_quantize():
    rng = np.random.default_rng(4)
    lens = np.array([17, 40, 1], dtype=np.int32)
    num_pages = 9
    bt = wl.permutation_block_tables(rng, lens, num_pages, 4)
    k_new = wl.bf16_normal_host(rng, (3, HKV, D))
    v_new = wl.bf16_normal_host(rng, (3, HKV, D))
    q = wl.bf16_normal_host(rng, (3, HQ, D))
    q_fp8, q_bf16 = q.copy(), q.copy()
    g = oracle.geom(num_pages)
    pool = fp8_pool(num_pages)
    before = pool.copy()
    oracle.append_fp8(pool, g, bt, lens - 1, k_new, v_new, q_fp8)
    ref = ph.new_pool(num_pages)
    oracle.append(ref, g, bt, lens - 1, k_new, v_new, q_bf16)
    assert np.array_equal(q_fp8, q_bf16)
    assert np.count_nonzero(pool != before) <= 3 * (2 * HKV * D + 2 * HKV * 4)
    pv = ph.Fp8Pages(pool)
    codes_v, scales_v = pv.codes(), pv.scales
    R = ph.pool_view(ref)
    for b in range(3):
        page, slot = bt[b, (lens[b] - 1) // PS], (lens[b] - 1) % PS
        for h in range(HKV):
            for kv in (0, 1):
                c, s = oracle.quantize_row_fp8(R[page, kv, h, slot])
                assert np.array_equal(codes_v[page, kv, h, slot], c) and scales_v[page, kv, h, slot] == s
    # head-major page: head 2's unit starts at 2 * 2176; K row 3 at 3 rows of 64; V slot 3 is the
    # odd slot of pair 1 (line 1 of 128 bytes), dim 4 in chunk 0, stored at chunk 0 ^ 2 = 2
    assert oracle.fp8_code_offset(g, 1, 0, 2, 3, 4) == PAGE + 2 * UNIT + 3 * D + 4
    assert oracle.fp8_code_offset(g, 1, 1, 2, 3, 4) == PAGE + 2 * UNIT + PS * D + 1 * 128 + 2 * 16 + 2 * 4 + 1
    assert oracle.fp8_code_offset(g, 0, 1, 0, 14, 63) == PS * D + 7 * 128 + (7 ^ 6) * 16 + 2 * 7 + 0
    assert oracle.fp8_scale_offset(g, 1, 1, 2, 3) == PAGE + 2 * UNIT + 2 * PS * D + (PS + 3) * 4
    assert UNIT == 2176
    unit_codes = {oracle.fp8_code_offset(g, 0, kv, 7, s, d) for kv in (0, 1) for s in range(PS) for d in range(D)}
    assert unit_codes == set(range(7 * UNIT, 7 * UNIT + 2 * PS * D))   # the codes fill their 2 KiB exactly
