"""Whole-layer parity at the benchmark's sizes and launch settings (GPU tests' helper).

``check_full_size`` builds a named workload with the launch configuration the
benchmark times (pages per unit, ring depth, dispatch order, micro-batch chains),
copies the pages of the layers to check from the device pool BEFORE the step, runs
one step from a captured CUDA graph, and then checks every (layer, sequence, query
head) of those layers against the oracle: the oracle appends the step's new token
to its own copy of the pages and decodes over them.  The oracle runs on the host
cores, one thread per slice of the batch (the C oracle releases the interpreter
lock; every sequence has its own pages, so the slices never write the same bytes).
Checked: every attention output within the parity tolerance, every rotated query
within one BF16 ulp, and the pages after the step against the oracle's (BF16:
placement and values bit-exact, keys within one ulp; FP8: value codes and scales
bit-exact, key rows within the quantization bound).
"""
import concurrent.futures
import math
import os

import numpy as np
import torch

import oracle
from paged_kv_decode_12_gb300 import harness, launch
from paged_kv_decode_12_gb300 import workloads as wl
from tests import paged_helpers as ph

SCALE = 1.0 / math.sqrt(wl.HEAD_DIM)
ATOL = RTOL = 1e-2


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def ulp_distance(a, b):
    def key(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)

    return np.abs(key(a) - key(b))


def snapshot_pages(dw, layers):
    """The pages of ``layers`` copied from the device pool into one compact host pool,
    and the layers' block tables renumbered into it: (pool bytes [pages][page_bytes] as
    uint8, bt [len(layers)][B][max_blocks], device page ids in compact order)."""
    w, eng = dw.w, dw.eng
    npg = -(-w.seq_lens.astype(np.int64) // wl.PAGE_SIZE)
    ids, bt = [], np.full((len(layers), w.batch, w.max_blocks), -1, dtype=np.int32)
    n = 0
    for i, l in enumerate(layers):
        for b in range(w.batch):
            row = eng.bt_host[l, b, :npg[b]]
            ids.append(row)
            bt[i, b, :npg[b]] = np.arange(n, n + npg[b], dtype=np.int32)
            n += int(npg[b])
    ids = np.concatenate(ids).astype(np.int64)
    return ids, bt


def gather(dw, ids) -> np.ndarray:
    view = dw.eng.slab.view(dw.eng.num_pages, dw.eng.page_bytes)
    out = np.empty((ids.size, dw.eng.page_bytes), dtype=np.uint8)
    step = 16384
    for s in range(0, ids.size, step):     # bounded device staging
        idx = torch.from_numpy(ids[s:s + step]).to(view.device)
        out[s:s + step] = view.index_select(0, idx).cpu().numpy()
    return out


def oracle_layer(kv, pool, bt, lens, q, k_new, v_new, threads):
    """Append + decode of one layer over ``pool`` (modified in place), on ``threads``
    host threads over slices of the batch: (out_f64 [B][32][64], rotated q [B][32][64])."""
    B = lens.size
    g = oracle.geom(pool.size // (oracle.FP8_PAGE_BYTES if kv == "fp8" else wl.PAGE_BYTES // 2))
    append, decode = (oracle.append_fp8, oracle.decode_fp8) if kv == "fp8" else (oracle.append, oracle.decode)
    q = q.copy()
    out = np.empty((B, wl.NUM_Q_HEADS, wl.HEAD_DIM), dtype=np.float64)

    def run(sl):
        qs = np.ascontiguousarray(q[sl])
        append(pool, g, bt[sl], lens[sl] - 1, k_new[sl], v_new[sl], qs)
        out[sl] = decode(pool, g, bt[sl], lens[sl], qs, SCALE)[1]
        q[sl] = qs

    bounds = np.linspace(0, B, min(B, threads) + 1).round().astype(int)
    slices = [slice(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(slices)) as ex:
        list(ex.map(run, slices))
    return out, q


def assert_close(got_u16, ref_f64, what):
    got = ph.bf16_to_f64(got_u16)
    err = np.abs(got - ref_f64)
    bound = ATOL + RTOL * np.abs(ref_f64)
    if not np.all(err <= bound):
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: max excess at {worst}: got {got[worst]} ref {ref_f64[worst]}")


def check_full_size(name, kv, layers):
    """The benchmark's configuration of workload ``name`` with ``kv`` pages, one step, every
    (sequence, query head) of ``layers`` checked against the oracle."""
    dw = harness.setup(name, **launch.config(name, kv))
    w = dw.w
    ids, bt = snapshot_pages(dw, layers)
    before = gather(dw, ids)
    # one eager step first (kernel attributes, tensor map): its appends write exactly the
    # bytes the timed step writes again, so the step below sees what a first step sees
    harness.warm(dw, 1)
    cap = harness.capture_steps(dw, 1)
    dw.reset_q()
    cap.graph.replay()
    torch.cuda.synchronize()
    st, flag = dw.eng.check_errors()
    assert st == 0 and flag == 0, (st, flag)
    after = gather(dw, ids)
    out, q_rot = u16(dw.out), u16(dw.q)
    q0, k_new, v_new = u16(dw.q0), u16(dw.k_new), u16(dw.v_new)
    lens = w.seq_lens.astype(np.int32)
    dw.eng.close()
    threads = os.cpu_count() or 1
    ref_pool = before.reshape(-1).copy()
    if kv == "bf16":
        ref_pool = ref_pool.view(np.uint16)
    for i, l in enumerate(layers):
        ref_out, ref_q = oracle_layer(kv, ref_pool, bt[i], lens, q0[l], k_new[l], v_new[l], threads)
        assert_close(out[l], ref_out, f"{name} {kv} layer {l}")
        assert ulp_distance(q_rot[l], ref_q).max() <= 1, f"rotated queries, layer {l}"
    ref = ref_pool.view(np.uint8).reshape(after.shape)
    if kv == "bf16":
        g_, r_, b_ = (x.reshape(-1).view(np.uint16) for x in (after, ref, before))
        assert np.array_equal(np.flatnonzero(g_ != b_), np.flatnonzero(r_ != b_))   # placement
        Pg, Pr = ph.pool_view(g_), ph.pool_view(r_)
        assert np.array_equal(Pg[:, 1], Pr[:, 1])                                      # values bit-exact
        assert ulp_distance(Pg[:, 0], Pr[:, 0]).max() <= 1                             # keys within one ulp
    else:
        # a page is 8 units of 2176 bytes, one per KV head: K code rows [16][64], V codes
        # (1024 bytes), K row scales [16], V row scales [16]; compared as raw bytes
        unit = oracle.FP8_PAGE_BYTES // wl.NUM_KV_HEADS
        kc, vc, ks = wl.PAGE_SIZE * wl.HEAD_DIM, 2 * wl.PAGE_SIZE * wl.HEAD_DIM, 2 * wl.PAGE_SIZE * wl.HEAD_DIM
        G, R = (x.reshape(-1, wl.NUM_KV_HEADS, unit) for x in (after, ref))
        assert np.array_equal(G[:, :, kc:vc], R[:, :, kc:vc])                           # value codes
        assert np.array_equal(G[:, :, ks + 64:], R[:, :, ks + 64:])                     # value scales
        written = np.zeros((G.shape[0], wl.NUM_KV_HEADS, wl.PAGE_SIZE), dtype=bool)   # appended key rows
        for i in range(len(layers)):
            for b, L in enumerate(lens):
                written[bt[i, b, (L - 1) // wl.PAGE_SIZE], :, (L - 1) % wl.PAGE_SIZE] = True
        Gk, Rk = (x[:, :, :kc].reshape(-1, wl.NUM_KV_HEADS, wl.PAGE_SIZE, wl.HEAD_DIM) for x in (G, R))
        Gs, Rs = (np.ascontiguousarray(x[:, :, ks:ks + 64]).view(np.float32) for x in (G, R))
        assert np.array_equal(Gk[~written], Rk[~written])
        assert np.array_equal(Gs[~written].view(np.uint32), Rs[~written].view(np.uint32))
        from tests.test_gpu_fp8 import assert_keys_close
        assert_keys_close(Gk[written], Gs[written], Rk[written], Rs[written])
    return w.batch * len(layers) * wl.NUM_Q_HEADS
