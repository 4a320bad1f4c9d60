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


# --------------------------------------------------------------------------- FP8 pages

_FP8_INDEX = None


def fp8_code_index(num_pages: int) -> np.ndarray:
    """Byte offsets [pages][2][8][16][64] of every code of an FP8 pool, from the oracle's
    layout function (the layout's one definition)."""
    import oracle

    global _FP8_INDEX
    if _FP8_INDEX is None:
        g = oracle.geom(1)
        idx = np.empty((2, wl.NUM_KV_HEADS, wl.PAGE_SIZE, wl.HEAD_DIM), dtype=np.int64)
        for kv in range(2):
            for h in range(wl.NUM_KV_HEADS):
                for s in range(wl.PAGE_SIZE):
                    for d in range(wl.HEAD_DIM):
                        idx[kv, h, s, d] = oracle.fp8_code_offset(g, 0, kv, h, s, d)
        _FP8_INDEX = idx
    page = oracle.FP8_PAGE_BYTES
    return _FP8_INDEX[None] + page * np.arange(num_pages, dtype=np.int64)[:, None, None, None, None]


class Fp8Pages:
    """Logical views of an FP8 pool's bytes: ``codes`` reads / writes the codes as
    [pages][2][8][16][64] (through the oracle's byte layout), ``scales`` is a float32 view
    [pages][2][8][16] of the row scales."""

    def __init__(self, pool: np.ndarray):
        import oracle

        self.pool = pool
        n = pool.size // oracle.FP8_PAGE_BYTES
        self.index = fp8_code_index(n)
        unit = oracle.FP8_PAGE_BYTES // wl.NUM_KV_HEADS
        codes_bytes = 2 * wl.PAGE_SIZE * wl.HEAD_DIM
        units = pool.reshape(n, wl.NUM_KV_HEADS, unit)
        self.scales = units[:, :, codes_bytes:].view(np.float32).reshape(n, wl.NUM_KV_HEADS, 2, wl.PAGE_SIZE)
        self.scales = self.scales.transpose(0, 2, 1, 3)

    def codes(self) -> np.ndarray:
        return self.pool[self.index]

    def set_row(self, page, kv, head, slot, codes, scale):
        self.pool[self.index[page, kv, head, slot]] = codes
        self.scales[page, kv, head, slot] = scale
