"""Pins for the oracle's paged decode attention and KV append.

Definitions (restated): scores are q.k scaled by 1/sqrt(head_dim), softmax with
the maximum subtracted, then the weighted sum of V ("从零构建大模型推理引擎", section
3.2); each query head streams its sequence's cached pages through the block
table (samir-vllm README summary, section "目前已完成的功能").

Pins, each able to catch a different plausible mistake:
  * L = 1 returns v_0 exactly                  (K/V swap, normalisation)
  * identical keys return the mean of V         (softmax normalisation)
  * weights are non-negative and sum to 1
  * paged == brute force over a contiguous cache (page / slot lookup)
  * contiguous == torch scaled_dot_product_attention in float64 with the KV
    heads repeated per group                      (scale, GQA map, transposes)
  * a dominating key returns its value, scores far beyond exp's FP64 range
                                                  (max subtraction)
  * physical page order does not change a single bit
  * append writes exactly the new token's K and V slots, V unrotated, K the
    rotated key within half a BF16 ulp, and the decode walk finds it there.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_12_gb300 import workloads as wl
from tests import paged_helpers as ph

HQ, HKV, D, PS = wl.NUM_Q_HEADS, wl.NUM_KV_HEADS, wl.HEAD_DIM, wl.PAGE_SIZE
SCALE = 1.0 / math.sqrt(D)


def _setup(seed, seq_lens, num_pages=None, max_blocks=8):
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B, S = len(seq_lens), int(seq_lens.max())
    num_pages = num_pages or ph.pages_needed(seq_lens) + 3
    K = wl.bf16_normal_host(rng, (B, HKV, S, D))
    V = wl.bf16_normal_host(rng, (B, HKV, S, D))
    q = wl.bf16_normal_host(rng, (B, HQ, D))
    bt = wl.permutation_block_tables(rng, seq_lens, num_pages, max_blocks)
    pool = ph.scatter_tokens(ph.new_pool(num_pages), bt, seq_lens, K, V)
    return dict(rng=rng, seq_lens=seq_lens, K=K, V=V, q=q, bt=bt, pool=pool,
                g=oracle.geom(num_pages))


def test_single_token_returns_v0_exactly():
    s = _setup(1, [1, 1, 1])
    out_bf16, out_f64 = oracle.decode(s["pool"], s["g"], s["bt"], s["seq_lens"], s["q"], SCALE)
    for b in range(3):
        for h in range(HQ):
            v0 = s["V"][b, h // 4, 0]
            assert np.array_equal(out_bf16[b, h], v0)
            assert np.array_equal(out_f64[b, h], ph.bf16_to_f64(v0))


def test_identical_keys_give_mean_of_values():
    s = _setup(2, [37])
    s["K"][0, :, :, :] = s["K"][0, :, :1, :]
    pool = ph.scatter_tokens(ph.new_pool(s["g"].num_pages), s["bt"], s["seq_lens"], s["K"], s["V"])
    _, out = oracle.decode(pool, s["g"], s["bt"], s["seq_lens"], s["q"], SCALE)
    for h in range(HQ):
        mean = ph.bf16_to_f64(s["V"][0, h // 4, :37]).mean(axis=0)
        assert np.allclose(out[0, h], mean, rtol=0, atol=1e-12)


def test_weights_sum_to_one():
    s = _setup(3, [53])
    for h in range(HQ):
        _, w = oracle.decode_one(s["pool"], s["g"], s["bt"][0], 53, s["q"][0, h], h // 4, SCALE,
                                 want_weights=True)
        assert np.all(w >= 0)
        assert abs(w.sum() - 1.0) <= 1e-12


def test_paged_equals_contiguous():
    lens = [1, 15, 16, 17, 40, 100]
    s = _setup(4, lens, max_blocks=7)
    _, paged = oracle.decode(s["pool"], s["g"], s["bt"], s["seq_lens"], s["q"], SCALE)
    contiguous = oracle.decode_contiguous(ph.bf16_to_f64(s["K"]), ph.bf16_to_f64(s["V"]),
                                          s["seq_lens"], ph.bf16_to_f64(s["q"]), SCALE)
    assert np.allclose(paged, contiguous, rtol=0, atol=1e-12)


def test_contiguous_equals_library_sdpa():
    lens = [3, 16, 33, 64]
    s = _setup(5, lens)
    K, V, q = (ph.bf16_to_f64(s[k]) for k in ("K", "V", "q"))
    ours = oracle.decode_contiguous(K, V, s["seq_lens"], q, SCALE)
    for b, L in enumerate(lens):
        kt = torch.from_numpy(K[b, :, :L]).repeat_interleave(HQ // HKV, dim=0)   # [HQ][L][D]
        vt = torch.from_numpy(V[b, :, :L]).repeat_interleave(HQ // HKV, dim=0)
        qt = torch.from_numpy(q[b]).unsqueeze(1)                                 # [HQ][1][D]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).squeeze(1).numpy()
        assert np.allclose(ours[b], ref, rtol=0, atol=1e-10)


def test_dominating_key_far_beyond_exp_range():
    s = _setup(6, [29])
    j, g = 11, 2
    # q for the group of KV head 2 is 400 x key j: its score is ~ 400*|k|^2/8 ~ 3200,
    # exp(3200) overflows FP64, so only a max-subtracted softmax stays finite.
    kj = ph.bf16_to_f64(s["K"][0, g, j])
    q = s["q"].copy()
    for h in range(4 * g, 4 * g + 4):
        q[0, h] = oracle.bf16_from_f64(400.0 * kj)
    _, out = oracle.decode(s["pool"], s["g"], s["bt"], s["seq_lens"], q, SCALE)
    assert np.all(np.isfinite(out))
    for h in range(4 * g, 4 * g + 4):
        assert np.allclose(out[0, h], ph.bf16_to_f64(s["V"][0, g, j]), rtol=0, atol=1e-12)


def test_physical_page_order_is_irrelevant():
    lens = [17, 40, 5]
    s = _setup(7, lens, num_pages=12)
    a_bf16, a = oracle.decode(s["pool"], s["g"], s["bt"], s["seq_lens"], s["q"], SCALE)
    bt2 = wl.permutation_block_tables(np.random.default_rng(99), lens, 12, s["bt"].shape[1])
    assert not np.array_equal(bt2, s["bt"])
    pool2 = ph.scatter_tokens(ph.new_pool(12), bt2, s["seq_lens"], s["K"], s["V"])
    b_bf16, b = oracle.decode(pool2, s["g"], bt2, s["seq_lens"], s["q"], SCALE)
    assert np.array_equal(a, b) and np.array_equal(a_bf16, b_bf16)


def test_gqa_groups_are_contiguous_query_heads():
    # change only KV head 5: query heads 20..23 and no others must move
    s = _setup(8, [21])
    _, before = oracle.decode(s["pool"], s["g"], s["bt"], s["seq_lens"], s["q"], SCALE)
    V = s["V"].copy()
    V[0, 5] = wl.bf16_normal_host(np.random.default_rng(5), V[0, 5].shape)
    pool = ph.scatter_tokens(ph.new_pool(s["g"].num_pages), s["bt"], s["seq_lens"], s["K"], V)
    _, after = oracle.decode(pool, s["g"], s["bt"], s["seq_lens"], s["q"], SCALE)
    moved = [h for h in range(HQ) if not np.array_equal(before[0, h], after[0, h])]
    assert moved == [20, 21, 22, 23]


def _half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    mag = np.maximum(np.abs(x), 2.0**-126)
    return 2.0 ** (np.floor(np.log2(mag)) - 8)


def test_append_placement_and_values():
    rng = np.random.default_rng(9)
    num_pages, max_blocks = 10, 6
    lens = np.array([17, 40, 1], dtype=np.int32)            # new tokens at positions 16, 39, 0
    pos = lens - 1
    bt = wl.permutation_block_tables(rng, lens, num_pages, max_blocks)
    g = oracle.geom(num_pages)
    pool = ph.new_pool(num_pages)
    k_new = wl.bf16_normal_host(rng, (3, HKV, D))
    v_new = wl.bf16_normal_host(rng, (3, HKV, D))
    q = wl.bf16_normal_host(rng, (3, HQ, D))
    q0 = q.copy()
    oracle.append(pool, g, bt, pos, k_new, v_new, q)

    changed = np.flatnonzero(pool != ph.SENTINEL)
    assert changed.size == 3 * 2 * HKV * D
    P = ph.pool_view(pool)
    for b in range(3):
        page, slot = bt[b, pos[b] // PS], pos[b] % PS
        assert np.array_equal(P[page, 1, :, slot, :], v_new[b])
        for kvh in range(HKV):
            x = ph.bf16_to_f64(k_new[b, kvh])
            i = np.arange(D // 2)
            freq = np.exp(-(2.0 * i / D) * math.log(wl.ROPE_THETA))
            z = (x[: D // 2] + 1j * x[D // 2:]) * np.exp(1j * int(pos[b]) * freq)
            exact = np.concatenate([z.real, z.imag])
            got = ph.bf16_to_f64(P[page, 0, kvh, slot, :])
            assert np.all(np.abs(got - exact) <= _half_ulp_bf16(exact))
        for h in range(HQ):
            x = ph.bf16_to_f64(q0[b, h])
            exact = oracle.rope_rotate(x, int(pos[b]), wl.ROPE_THETA)
            assert np.all(np.abs(ph.bf16_to_f64(q[b, h]) - exact) <= _half_ulp_bf16(exact))
    if pos[2] == 0:
        assert np.array_equal(q[2], q0[2])  # position 0 leaves q unchanged


def test_append_then_decode_finds_the_new_token():
    rng = np.random.default_rng(10)
    lens = np.array([18], dtype=np.int32)                   # new token at position 17 (page 1, slot 1)
    num_pages = 4
    bt = wl.permutation_block_tables(rng, lens, num_pages, 4)
    K = wl.bf16_normal_host(rng, (1, HKV, 18, D))
    V = wl.bf16_normal_host(rng, (1, HKV, 18, D))
    pool = ph.scatter_tokens(ph.new_pool(num_pages), bt, lens - 1, K, V)   # 17 cached tokens
    g = oracle.geom(num_pages)
    k_new = wl.bf16_normal_host(rng, (1, HKV, D))
    v_new = wl.bf16_normal_host(rng, (1, HKV, D))
    # q = 100 k_new for every head of group 0: after both are rotated to the same
    # position the new token's score dominates and the output is v_new.
    q = np.zeros((1, HQ, D), dtype=np.uint16)
    for h in range(HQ):
        q[0, h] = oracle.bf16_from_f64(100.0 * ph.bf16_to_f64(k_new[0, h // 4]))
    oracle.append(pool, g, bt, lens - 1, k_new, v_new, q)
    _, out = oracle.decode(pool, g, bt, lens, q, SCALE)
    for h in range(HQ):
        assert np.allclose(out[0, h], ph.bf16_to_f64(v_new[0, h // 4]), rtol=0, atol=1e-9)


def test_rejects_bad_inputs():
    s = _setup(11, [20])
    bad = s["bt"].copy()
    bad[0, 1] = s["g"].num_pages            # out-of-range page id
    with pytest.raises(oracle.OracleError):
        oracle.decode(s["pool"], s["g"], bad, s["seq_lens"], s["q"], SCALE)
    with pytest.raises(oracle.OracleError):
        oracle.decode(s["pool"], s["g"], s["bt"], np.array([0], dtype=np.int32), s["q"], SCALE)
