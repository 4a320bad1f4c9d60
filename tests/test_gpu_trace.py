"""GPU parity of the prefill page fill and of decode steps inside a scheduler-driven
continuous-batching trace.

* pkv_prefill_append writes exactly the oracle's bytes (positions bit-exact, V
  bit-exact, K within 1 BF16 ulp), the oracle's append applied token by token;
* during a trace (admission by page budget, prefill, lazy pages, retirement),
  sampled outputs of several steps match the oracle computed on a snapshot of the
  sequence's pages taken just before the step.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300 import workloads as wl
from paged_kv_decode_12_gb300.trace import TraceRunner
from tests import paged_helpers as ph
from tests.test_gpu_parity import assert_close, dev_bf16, u16, ulp_distance

pytestmark = pytest.mark.gpu

HKV, D, PS = wl.NUM_KV_HEADS, wl.HEAD_DIM, wl.PAGE_SIZE


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


@pytest.mark.parametrize("start,T", [(0, 37), (5, 16), (30, 100)])
def test_prefill_fill_matches_oracle(start, T):
    rng = np.random.default_rng(start + T)
    layers, max_blocks, num_pages = 3, 16, 64
    L = start + T
    bt = np.full((layers, max_blocks), -1, dtype=np.int32)
    perm = rng.permutation(num_pages).astype(np.int32)
    npg = math.ceil(L / PS)
    for layer in range(layers):
        bt[layer, :npg] = perm[layer * npg:(layer + 1) * npg]
    k = wl.bf16_normal_host(rng, (layers, T, HKV, D))
    v = wl.bf16_normal_host(rng, (layers, T, HKV, D))
    pool0 = ph.new_pool(num_pages)
    slab = torch.from_numpy(pool0.view(np.uint8).copy()).cuda()
    p = pkv.pkv_pool_create(slab, slab.numel())
    rope = torch.empty(2048 * D, dtype=torch.float32, device="cuda")
    pkv.pkv_rope_table_init(wl.ROPE_THETA, 2048, D // 2, rope)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_prefill_append(p, dev_bf16(k), dev_bf16(v), torch.from_numpy(bt).cuda(), max_blocks, layers, start, T,
                           rope, 2048, err)
    st, flag = pkv.pkv_check_device_error(err)
    assert st == pkv.PKV_OK and flag == 0
    got = u16(slab.view(torch.bfloat16))
    ref = pool0.copy()
    g = oracle.geom(num_pages)
    for layer in range(layers):
        rows = np.repeat(bt[layer][None], T, axis=0)
        oracle.append(ref, g, rows, np.arange(start, L, dtype=np.int32), k[layer], v[layer])
    assert np.array_equal(np.flatnonzero(got != pool0), np.flatnonzero(ref != pool0))
    P_g, P_r = ph.pool_view(got), ph.pool_view(ref)
    assert np.array_equal(P_g[:, 1], P_r[:, 1])                       # values bit-exact
    assert ulp_distance(P_g[:, 0], P_r[:, 0]).max() <= 1              # rotated keys within 1 ulp
    pkv.pkv_pool_destroy(p)


def test_trace_steps_match_oracle():
    layers, max_batch = 2, 24
    runner = TraceRunner(pool_pages=3000, layers=layers, max_batch=max_batch, pages_per_chunk=4, seed=5)
    reqs = wl.trace_schedule(seed=5, steps=60, arrival_rate=0.8, prompt_lo=8, prompt_hi=200, out_lo=4, out_hi=60)
    rng = np.random.default_rng(9)
    check_steps = {3, 17, 31, 45, 59}
    pending = {}

    def before(step, ids, lens, bt):
        if step not in check_steps:
            return
        picks = []
        for _ in range(4):
            b = int(rng.integers(ids.size))
            layer = int(rng.integers(layers))
            h = int(rng.integers(wl.NUM_Q_HEADS))
            L = int(lens[b])
            npg = math.ceil(L / PS)
            pages = torch.from_numpy(bt[layer, b, :npg].astype(np.int64)).cuda()
            pool_view = runner.slab.view(torch.bfloat16).view(runner.num_pages, 2, HKV, PS, D)
            picks.append(dict(b=b, layer=layer, h=h, L=L, npg=npg, mini=u16(pool_view[pages]).reshape(-1).copy(),
                              q=u16(runner.q[layer, b]).copy(), k=u16(runner.k_new[layer, b]).copy(),
                              v=u16(runner.v_new[layer, b]).copy()))
        pending[step] = picks

    def after(step, ids, lens, bt):
        if step not in pending:
            return
        torch.cuda.synchronize()
        out = u16(runner.out)
        for pk in pending.pop(step):
            g = oracle.geom(pk["npg"])
            row = np.full((1, runner.max_blocks), -1, dtype=np.int32)
            row[0, :pk["npg"]] = np.arange(pk["npg"])
            q = pk["q"][None].copy()
            oracle.append(pk["mini"], g, row, [pk["L"] - 1], pk["k"][None], pk["v"][None], q)
            ref = oracle.decode_one(pk["mini"], g, row[0], pk["L"], q[0, pk["h"]], pk["h"] // 4, runner.scale)
            assert_close(out[pk["layer"], pk["b"], pk["h"]], ref)

    res = runner.run(reqs, 60, before, after)
    assert not pending
    st, flag = pkv.pkv_check_device_error(runner.err)
    assert st == pkv.PKV_OK and flag == 0
    s = res.stats
    assert s["max_decode_batch"] == max(res.batch_sizes) and s["peak_active"] >= s["max_decode_batch"]
    assert s["allocated_pages"] + s["final_free_pages"] == s["pool_pages"]
    assert res.decode_steps > 0 and res.tokens == sum(res.batch_sizes)
    runner.close()
