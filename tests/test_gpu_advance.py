"""GPU parity over consecutive decode steps whose positions advance.

Every step appends one token per sequence at position seq_len - 1 and attends over
the pages including it; the next step's sequences are one token longer.  The steps
run back to back from one CUDA graph, with programmatic dependent launch, so each
launch overlaps the tail of the one before it.  With one layer, the launch before a
step's launch is the previous step of the same layer, which wrote position
seq_len - 2 of every sequence: the page holding it must be read only after the
dependency wait, or the step would attend over stale bytes.  Lengths cross page
boundaries (15 -> 55, 1 -> 41, ...), so that position sometimes sits in the
previous page.

Checked against the oracle run step by step (samir-vllm README summary, "目前已完成的
功能": decode appends one token at its absolute RoPE position, and later steps attend
to it): every step's outputs within the parity tolerance and its rotated queries
within one BF16 ulp; after the last step, the pool holds exactly the oracle's
cumulative appends (placement and values bit-exact, keys within one BF16 ulp; FP8:
codes of values and scales bit-exact, key rows within the quantization bound).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300 import workloads as wl
from paged_kv_decode_12_gb300.engine import DecodeEngine
from tests import paged_helpers as ph
from tests import test_gpu_fp8 as f8
from tests.test_gpu_parity import assert_close, dev_bf16, make_case, u16, ulp_distance

pytestmark = pytest.mark.gpu

HQ, HKV, D, PS = wl.NUM_Q_HEADS, wl.NUM_KV_HEADS, wl.HEAD_DIM, wl.PAGE_SIZE
SCALE = 1.0 / math.sqrt(D)
STEPS = 41
START = np.array([15, 1, 16, 31, 2, 47], dtype=np.int32)   # lengths at the first step


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def build_case(kv, layers, seed):
    """A pool whose tables hold pages for the final lengths of every (layer, sequence),
    with positions below the first step's new token filled (the rest gets overwritten
    by the appends); per-step seeded q, k_new, v_new."""
    B = START.size
    final = START + STEPS - 1
    lens = np.tile(final, layers)                       # one row per (layer, sequence)
    max_blocks = -(-int(final.max()) // PS) + 1
    c = (f8.make_case if kv == "fp8" else make_case)(seed, lens, max_blocks=max_blocks)
    bt = c["bt"].reshape(layers, B, max_blocks)
    rng = np.random.default_rng(seed + 1)
    q = wl.bf16_normal_host(rng, (STEPS, layers, B, HQ, D))
    k = wl.bf16_normal_host(rng, (STEPS, layers, B, HKV, D))
    v = wl.bf16_normal_host(rng, (STEPS, layers, B, HKV, D))
    lens_steps = np.stack([START + s for s in range(STEPS)]).astype(np.int32)
    return dict(pool=c["pool"], bt=bt, num_pages=c["num_pages"], max_blocks=max_blocks, q=q, k=k, v=v,
                lens=lens_steps, B=B, layers=layers)


def run_gpu(c, kv, fused, sorted_units, chunk):
    eng = DecodeEngine(c["num_pages"], c["layers"], c["B"], c["max_blocks"], chunk, kv=kv, fused=fused,
                       sorted_units=sorted_units)
    pool0 = torch.from_numpy(c["pool"].view(np.uint8).copy()).cuda()
    eng.slab.copy_(pool0)
    eng.set_tables(c["bt"])
    q = dev_bf16(c["q"])
    k, v = dev_bf16(c["k"]), dev_bf16(c["v"])
    lens = torch.from_numpy(c["lens"]).cuda()
    pos = (lens - 1).contiguous()
    out = torch.zeros_like(q)
    # one eager step first (kernel attributes, tensor map), then the state is restored
    eng.step(q[0].clone(), k[0], v[0], pos[0], lens[0], out[0].clone())
    torch.cuda.synchronize()
    eng.slab.copy_(pool0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for s in range(STEPS):   # back to back: each launch may overlap the previous one
            eng.step(q[s], k[s], v[s], pos[s], lens[s], out[s])
    graph.replay()
    torch.cuda.synchronize()
    st, flag = eng.check_errors()
    slab = eng.slab.cpu().numpy()
    res = dict(status=st, flag=flag, out=u16(out), q=u16(q), slab=slab.view(np.uint16) if kv == "bf16" else slab)
    eng.close()
    return res


@pytest.mark.parametrize("kv,layers,sched,path,chunk", [
    ("bf16", 1, "grid", "fused", 1),
    ("bf16", 1, "grid", "fused", 3),
    ("bf16", 1, "sorted", "fused", 1),
    ("bf16", 2, "grid", "fused", 2),
    ("bf16", 1, "grid", "separate", 1),
    ("fp8", 1, "grid", "fused", 1),
    ("fp8", 1, "sorted", "fused", 3),
    ("fp8", 2, "grid", "fused", 2),
    ("fp8", 1, "grid", "separate", 2),
])
def test_steps_with_advancing_positions_match_oracle(kv, layers, sched, path, chunk):
    c = build_case(kv, layers, seed=80 + layers + (10 if kv == "fp8" else 0))
    gpu = run_gpu(c, kv, path == "fused", sched == "sorted", chunk)
    assert gpu["status"] == pkv.PKV_OK and gpu["flag"] == 0
    pool = c["pool"].copy()
    g = oracle.geom(c["num_pages"])
    append, decode = (oracle.append_fp8, oracle.decode_fp8) if kv == "fp8" else (oracle.append, oracle.decode)
    for s in range(STEPS):
        for layer in range(layers):
            q = c["q"][s, layer].copy()
            append(pool, g, c["bt"][layer], c["lens"][s] - 1, c["k"][s, layer], c["v"][s, layer], q)
            _, ref = decode(pool, g, c["bt"][layer], c["lens"][s], q, SCALE)
            assert_close(gpu["out"][s, layer], ref)
            assert ulp_distance(gpu["q"][s, layer], q).max() <= 1, (s, layer)
    # the pool after the last step: the oracle's cumulative appends
    if kv == "bf16":
        assert np.array_equal(np.flatnonzero(gpu["slab"] != c["pool"]), np.flatnonzero(pool != c["pool"]))
        Pg, Po = ph.pool_view(gpu["slab"]), ph.pool_view(pool)
        assert np.array_equal(Pg[:, 1], Po[:, 1])                        # values bit-exact
        assert ulp_distance(Pg[:, 0], Po[:, 0]).max() <= 1               # keys within one ulp
    else:
        gc, gs = f8.views(gpu["slab"])
        rc, rs = f8.views(pool)
        assert np.array_equal(gc[:, 1], rc[:, 1])                        # value codes bit-exact
        assert np.array_equal(gs[:, 1].view(np.uint32), rs[:, 1].view(np.uint32))
        written = np.zeros(gc.shape[:1] + gc.shape[2:4], dtype=bool)     # [page][head][slot] of appended keys
        for layer in range(layers):
            for b in range(c["B"]):
                for L in c["lens"][:, b]:
                    written[c["bt"][layer, b, (L - 1) // PS], :, (L - 1) % PS] = True
        keys_g, keys_r = gc[:, 0], rc[:, 0]
        assert np.array_equal(keys_g[~written], keys_r[~written])
        assert np.array_equal(gs[:, 0][~written].view(np.uint32), rs[:, 0][~written].view(np.uint32))
        f8.assert_keys_close(keys_g[written], gs[:, 0][written], keys_r[written], rs[:, 0][written])
