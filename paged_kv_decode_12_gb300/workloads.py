"""Seeded synthetic workloads for the paged-KV decode path.

This module only draws inputs: sequence lengths, block-table permutations and
N(0,1) values rounded to BF16 by the framework's own dtype conversion.  It holds
none of the method's arithmetic, so both the CUDA path (through the bench and
the GPU tests) and the CPU oracle (through the tests) can use it.

Workloads follow the engine's shapes: Llama-3.2-1B attention (32 query heads,
8 KV heads, head_dim 64), 16-token pages, a 2,048-token context cap, 16 layers.
The five named shapes are:

``tiny``  1 layer, lengths {17, 40}, an 8-page pool, block tables a seeded
          random permutation of the pool's pages.
``b8``    16 layers, batch 8, lengths uniform in [1, 2048], 4,096 pages of
          32 KiB per layer (65,536 pages, 2 GiB).
``b64``   16 layers, batch 64, log-normal lengths (median 300, sigma 1.0,
          clipped to [1, 2048]); the first six draws are replaced by
          1, 16, 17, 32, 33, 2048 so every page boundary case occurs; 1 % of
          the (token, KV head) key rows are multiplied by 8; same pool as b8.
``b256``  16 layers, batch 256, every length 2048 (128 pages per sequence and
          layer), 524,288 pages (16 GiB).
``trace`` the continuous-batching arrival schedule (see ``trace_schedule``).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PAGE_SIZE = 16
NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
MAX_CONTEXT = 2048
MAX_BLOCKS = MAX_CONTEXT // PAGE_SIZE          # 128 logical pages per (sequence, layer)
PAGE_BYTES = 2 * NUM_KV_HEADS * PAGE_SIZE * HEAD_DIM * 2   # K and V, BF16: 32 KiB
ROPE_THETA = 500000.0
DEFAULT_SEED = 12


PAGE_BYTES_FP8 = 2 * NUM_KV_HEADS * PAGE_SIZE * (HEAD_DIM + 4)   # E4M3 codes + FP32 row scales: 17 KiB


def kv_bytes_per_token(layers: int, kv_heads: int = NUM_KV_HEADS, head_dim: int = HEAD_DIM,
                       elem_bytes: int = 2, kv: str = "bf16") -> int:
    """KV-cache bytes one token adds: K and V, every layer and KV head (FP8 pages:
    one code byte per value plus a 4-byte scale per row)."""
    if kv == "fp8":
        return 2 * layers * kv_heads * (head_dim + 4)
    return 2 * layers * kv_heads * head_dim * elem_bytes


@dataclasses.dataclass
class Workload:
    name: str
    layers: int
    seq_lens: np.ndarray            # int32 [B], post-append lengths (position = length - 1)
    pool_pages: int                 # pages in the whole slab, all layers
    key_outlier_frac: float = 0.0   # fraction of key rows scaled by 8
    seed: int = DEFAULT_SEED
    max_blocks: int = MAX_BLOCKS

    @property
    def batch(self) -> int:
        return int(self.seq_lens.size)

    @property
    def positions(self) -> np.ndarray:
        return (self.seq_lens - 1).astype(np.int32)

    def kv_bytes_per_step(self, kv: str = "bf16") -> int:
        """KV bytes read by one pass over all layers: every cached token's K and V once."""
        return int(self.seq_lens.astype(np.int64).sum()) * kv_bytes_per_token(self.layers, kv=kv)

    def pages_per_layer(self) -> int:
        return int(sum(math.ceil(int(L) / PAGE_SIZE) for L in self.seq_lens))


def lognormal_lengths(rng: np.random.Generator, n: int, median: float = 300.0, sigma: float = 1.0,
                      lo: int = 1, hi: int = MAX_CONTEXT) -> np.ndarray:
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


def make_workload(name: str, seed: int = DEFAULT_SEED) -> Workload:
    rng = np.random.default_rng(seed)
    if name == "tiny":
        return Workload("tiny", 1, np.array([17, 40], dtype=np.int32), pool_pages=8, seed=seed)
    if name == "b8":
        lens = rng.integers(1, MAX_CONTEXT, size=8, endpoint=True).astype(np.int32)
        return Workload("b8", 16, lens, pool_pages=4096 * 16, seed=seed)
    if name == "b64":
        lens = lognormal_lengths(rng, 64)
        lens[:6] = [1, 16, 17, 32, 33, 2048]
        return Workload("b64", 16, lens, pool_pages=4096 * 16, key_outlier_frac=0.01, seed=seed)
    if name == "b256":
        lens = np.full(256, MAX_CONTEXT, dtype=np.int32)
        return Workload("b256", 16, lens, pool_pages=256 * MAX_BLOCKS * 16, seed=seed)
    raise ValueError(f"unknown workload {name!r}")


WORKLOADS = ("tiny", "b8", "b64", "b256")


# --------------------------------------------------------------------------- host draws

def bf16_normal_host(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) FP32 draws rounded to BF16 by torch's dtype conversion; returns uint16 bits."""
    import torch

    x = rng.standard_normal(size=shape, dtype=np.float32)
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def scale_bf16_by_8(bits: np.ndarray) -> np.ndarray:
    """Multiply BF16 values by 8 (exact: the exponent grows by 3) through torch."""
    import torch

    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return (t * 8).view(torch.int16).numpy().view(np.uint16).copy()


def permutation_block_tables(rng: np.random.Generator, seq_lens, num_pages: int,
                             max_blocks: int = MAX_BLOCKS) -> np.ndarray:
    """Block tables [B][max_blocks] drawn from one random permutation of the pool's pages.

    Unused entries are -1.  Raises if the pool is too small.
    """
    need = [math.ceil(int(L) / PAGE_SIZE) for L in seq_lens]
    if sum(need) > num_pages:
        raise ValueError("pool too small for these lengths")
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt


# --------------------------------------------------------------------------- device draws

def fill_bf16_normal_(t, seed: int, chunk_elems: int = 1 << 28):
    """Fill a CUDA bfloat16 tensor in place with seeded N(0,1) draws, chunk by chunk."""
    import torch

    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    flat = t.view(-1)
    for start in range(0, flat.numel(), chunk_elems):
        stop = min(start + chunk_elems, flat.numel())
        flat[start:stop].copy_(torch.randn(stop - start, generator=g, device=t.device,
                                           dtype=torch.float32))
    return t


def scale_key_rows_(pool_bf16, frac: float, seed: int):
    """Multiply a random ``frac`` of (page, KV head, slot) key rows by 8, in place.

    ``pool_bf16`` is the slab viewed as [pages][2][Hkv][P][D] bfloat16.
    """
    import torch

    if frac <= 0:
        return pool_bf16
    g = torch.Generator(device=pool_bf16.device)
    g.manual_seed(seed)
    pages = pool_bf16.shape[0]
    step = 4096
    for p0 in range(0, pages, step):
        p1 = min(p0 + step, pages)
        mask = torch.rand((p1 - p0, NUM_KV_HEADS, PAGE_SIZE), generator=g,
                          device=pool_bf16.device) < frac
        keys = pool_bf16[p0:p1, 0]
        keys.mul_(torch.where(mask, 8.0, 1.0).to(keys.dtype).unsqueeze(-1))
    return pool_bf16


def fill_fp8_pages_(codes, scales, seed: int, key_outlier_frac: float = 0.0):
    """Fill an FP8 pool's codes (uint8 [pages][2][Hkv][P][D]) and row scales (float32
    [pages][2][Hkv][P]) in place with seeded draws shaped like quantized N(0,1) rows:
    codes are N(0, 128^2) draws converted to E4M3 by torch's float8_e4m3fn dtype
    (clamped to +-448 first), scales uniform in [0.005, 0.009] (about 3/448, the
    scale of a 64-value N(0,1) row).  A ``key_outlier_frac`` share of key rows get
    8x scales."""
    import torch

    g = torch.Generator(device=codes.device)
    g.manual_seed(seed)
    pages = codes.shape[0]
    step = 4096
    for p0 in range(0, pages, step):
        p1 = min(p0 + step, pages)
        x = torch.randn(codes[p0:p1].shape, generator=g, device=codes.device, dtype=torch.float32) * 128.0
        codes[p0:p1].copy_(x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
        u = torch.rand(scales[p0:p1].shape, generator=g, device=codes.device, dtype=torch.float32)
        s = 0.005 + 0.004 * u
        if key_outlier_frac > 0:
            mask = torch.rand((p1 - p0, NUM_KV_HEADS, PAGE_SIZE), generator=g, device=codes.device) < key_outlier_frac
            s[:, 0] = torch.where(mask, s[:, 0] * 8.0, s[:, 0])
        scales[p0:p1].copy_(s)
    return codes, scales


# --------------------------------------------------------------------------- trace

@dataclasses.dataclass
class TraceRequest:
    rid: int
    arrival_step: int
    prompt_len: int
    max_new: int


def trace_schedule(seed: int = DEFAULT_SEED, steps: int = 500, arrival_rate: float = 0.6,
                   prompt_lo: int = 8, prompt_hi: int = 1024, out_lo: int = 16,
                   out_hi: int = 1024) -> list:
    """Seeded arrivals for the continuous-batching trace: Poisson(arrival_rate) per step,
    prompt lengths U[prompt_lo, prompt_hi], output budgets U[out_lo, out_hi]."""
    rng = np.random.default_rng(seed)
    reqs = []
    rid = 0
    for step in range(steps):
        for _ in range(int(rng.poisson(arrival_rate))):
            p = int(rng.integers(prompt_lo, prompt_hi, endpoint=True))
            o = int(rng.integers(out_lo, out_hi, endpoint=True))
            reqs.append(TraceRequest(rid, step, p, o))
            rid += 1
    return reqs
