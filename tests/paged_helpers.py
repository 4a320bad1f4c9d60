"""Test-side helpers: lay logical K/V rows into a page pool, and read them back.

The pool layout is the library's documented one: a slab of pages, each page
[2 (K, V)][Hkv][page_size][head_dim] BF16.  These helpers express it with numpy
indexing, independently of both the oracle's index function and the CUDA code,
so that tests can build paged inputs from contiguous ones and back.
"""
import math

import numpy as np

from paged_kv_decode_12_gb300 import workloads as wl

SENTINEL = 0xFFFF  # a NaN pattern no N(0,1) draw produces


def pool_view(pool_flat: np.ndarray, page_size=wl.PAGE_SIZE, hkv=wl.NUM_KV_HEADS, d=wl.HEAD_DIM):
    return pool_flat.reshape(-1, 2, hkv, page_size, d)


def new_pool(num_pages: int, fill=SENTINEL) -> np.ndarray:
    return np.full(num_pages * 2 * wl.NUM_KV_HEADS * wl.PAGE_SIZE * wl.HEAD_DIM, fill, dtype=np.uint16)


def scatter_tokens(pool_flat, bt, seq_lens, K, V):
    """Write logical rows K[b][g][t], V[b][g][t] (t < L_b) to their page slots."""
    P = pool_view(pool_flat)
    ps = P.shape[3]
    for b, L in enumerate(seq_lens):
        for t in range(int(L)):
            page = bt[b, t // ps]
            P[page, 0, :, t % ps, :] = K[b, :, t, :]
            P[page, 1, :, t % ps, :] = V[b, :, t, :]
    return pool_flat


def gather_tokens(pool_flat, bt_row, L):
    """Read back logical K, V rows [Hkv][L][D] of one sequence."""
    P = pool_view(pool_flat)
    ps = P.shape[3]
    pages = np.array([bt_row[t // ps] for t in range(L)])
    slots = np.arange(L) % ps
    K = P[pages, 0, :, slots, :].transpose(1, 0, 2)
    V = P[pages, 1, :, slots, :].transpose(1, 0, 2)
    return K, V


def pages_needed(seq_lens, page_size=wl.PAGE_SIZE):
    return sum(math.ceil(int(L) / page_size) for L in seq_lens)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bits -> float64 through numpy bit manipulation (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
