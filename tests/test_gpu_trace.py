"""GPU parity of the prefill page fill and of decode steps inside a scheduler-driven
continuous-batching trace.

* pkv_prefill_append writes exactly the oracle's bytes (positions bit-exact, V
  bit-exact, K within 1 BF16 ulp), the oracle's append applied token by token;
* during a trace (admission by page budget, prefill, lazy pages, retirement),
  sampled outputs of several steps match the oracle, which rebuilds the sequence's
  pages from the raw seeded inputs (prompt draw, each step's new K/V row), for BF16
  and FP8 pages.
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
    rope = pkv.rope_table(2048, "cuda", wl.ROPE_THETA)
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


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_prefill_then_decode_back_to_back(kv):
    # prompts filled by pkv_prefill_append and decoded right after, every launch in one
    # CUDA graph with no other work between them: the decode launch after a prefill on the
    # pool must not read the prompt pages before the prefill has finished
    from paged_kv_decode_12_gb300.engine import DecodeEngine

    rng = np.random.default_rng(41)
    prompts = np.array([30, 17, 64, 5, 1, 48], dtype=np.int32)
    B, layers, max_blocks = prompts.size, 1, 8
    lens = prompts + 1
    eng = DecodeEngine(B * max_blocks + 4, layers, B, max_blocks, pages_per_chunk=1, kv=kv)
    bt = eng.build_tables(lens)
    k = [wl.bf16_normal_host(rng, (layers, int(T), HKV, D)) for T in prompts]
    v = [wl.bf16_normal_host(rng, (layers, int(T), HKV, D)) for T in prompts]
    q = wl.bf16_normal_host(rng, (layers, B, wl.NUM_Q_HEADS, D))
    k_new = wl.bf16_normal_host(rng, (layers, B, HKV, D))
    v_new = wl.bf16_normal_host(rng, (layers, B, HKV, D))
    kd, vd = [dev_bf16(x) for x in k], [dev_bf16(x) for x in v]
    rows = [torch.from_numpy(np.ascontiguousarray(bt[:, b])).cuda() for b in range(B)]
    qd, knd, vnd = dev_bf16(q), dev_bf16(k_new), dev_bf16(v_new)
    lens_d = torch.from_numpy(lens).cuda()
    out = torch.zeros_like(qd)
    slab0 = eng.slab.clone()
    # first pass eager (kernel attributes, tensor map), then restore and replay from a graph
    for b in range(B):
        pkv.pkv_prefill_append(eng.pool, kd[b], vd[b], rows[b], max_blocks, layers, 0, int(prompts[b]), eng.rope,
                               eng.max_pos, eng.err)
    eng.step(qd.clone(), knd, vnd, lens_d - 1, lens_d, out.clone())
    torch.cuda.synchronize()
    eng.slab.copy_(slab0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for b in range(B):
            pkv.pkv_prefill_append(eng.pool, kd[b], vd[b], rows[b], max_blocks, layers, 0, int(prompts[b]),
                                   eng.rope, eng.max_pos, eng.err)
        eng.step(qd, knd, vnd, lens_d - 1, lens_d, out)
    g.replay()
    torch.cuda.synchronize()
    st, flag = eng.check_errors()
    assert st == pkv.PKV_OK and flag == 0
    got = u16(out)
    eng.close()
    fp8 = kv == "fp8"
    append = oracle.append_fp8 if fp8 else oracle.append
    decode_one = oracle.decode_one_fp8 if fp8 else oracle.decode_one
    for b in range(B):
        L = int(lens[b])
        npg = math.ceil(L / PS)
        gg = oracle.geom(npg)
        row = np.full((1, max_blocks), -1, dtype=np.int32)
        row[0, :npg] = np.arange(npg)
        mini = np.zeros(npg * oracle.FP8_PAGE_BYTES, np.uint8) if fp8 else ph.new_pool(npg)
        for t in range(L - 1):
            append(mini, gg, row, [t], k[b][0, t][None], v[b][0, t][None])
        qq = q[0, b][None].copy()
        append(mini, gg, row, [L - 1], k_new[0, b][None], v_new[0, b][None], qq)
        for h in range(wl.NUM_Q_HEADS):
            assert_close(got[0, b, h], decode_one(mini, gg, row[0], L, qq[0, h], h // 4, 1.0 / math.sqrt(D)))


@pytest.mark.parametrize("kv,chains,static", [("bf16", 1, False), ("fp8", 1, False), ("bf16", 3, False),
                                               ("bf16", 1, True), ("fp8", 1, True)])
def test_trace_steps_match_oracle(kv, chains, static):
    # The oracle rebuilds each sampled sequence's pages from the raw seeded inputs that
    # went into them -- the prompt K/V draw of its admission and the new K/V row of every
    # step since -- and decodes with the step's unrotated query; nothing the CUDA path
    # wrote is read back as an oracle input.  Static batching (samir-vllm README summary,
    # "构建": --static; "当前范围": the next group is admitted only after the current one
    # has finished) runs the same kernels on group-wise batches.
    layers, max_batch = 2, 24
    runner = TraceRunner(pool_pages=3000, layers=layers, max_batch=max_batch, pages_per_chunk=4, seed=5, kv=kv,
                         chains=chains, static=static)
    fp8 = kv == "fp8"
    # static groups live as long as their longest member: shorter budgets let several groups run
    reqs = wl.trace_schedule(seed=5, steps=60, arrival_rate=0.8, prompt_lo=8, prompt_hi=200, out_lo=4,
                             out_hi=25 if static else 60)
    rng = np.random.default_rng(9)
    check_steps = {3, 17, 31, 45, 59}
    k_new, v_new, q0 = u16(runner.k_new), u16(runner.v_new), u16(runner.q0)
    history = {}   # request id -> [(position, batch slot)] of its decode tokens so far
    pending = {}
    batches = []   # the ids of every non-empty decode batch, in step order

    def before(step, ids, lens, bt):
        batches.append(set(ids.tolist()))
        for b, rid in enumerate(ids.tolist()):
            history.setdefault(rid, []).append((int(lens[b]) - 1, b))
        if step in check_steps:
            pending[step] = [(int(rng.integers(ids.size)), int(rng.integers(layers)), int(rng.integers(wl.NUM_Q_HEADS)),
                              ids.copy(), lens.copy()) for _ in range(4)]

    def oracle_out(rid, L, layer, b, h):
        seed, plen = runner.prompt_seeds[rid]
        kp, vp = runner.prompt_kv(seed, plen)
        k = np.concatenate([u16(kp)[layer], np.stack([k_new[layer, s] for _, s in history[rid]])])
        v = np.concatenate([u16(vp)[layer], np.stack([v_new[layer, s] for _, s in history[rid]])])
        assert k.shape[0] == L and [p for p, _ in history[rid]] == list(range(plen, L))
        npg = math.ceil(L / PS)
        g = oracle.geom(npg)
        row = np.full((1, runner.max_blocks), -1, dtype=np.int32)
        row[0, :npg] = np.arange(npg)
        mini = np.zeros(npg * oracle.FP8_PAGE_BYTES, np.uint8) if fp8 else ph.new_pool(npg)
        append = oracle.append_fp8 if fp8 else oracle.append
        for pos in range(L - 1):
            append(mini, g, row, [pos], k[pos][None], v[pos][None])
        q = q0[layer, b][None].copy()
        append(mini, g, row, [L - 1], k[L - 1][None], v[L - 1][None], q)
        decode_one = oracle.decode_one_fp8 if fp8 else oracle.decode_one
        return decode_one(mini, g, row[0], L, q[0, h], h // 4, runner.scale)

    def after(step, ids, lens, bt):
        if step not in pending:
            return
        torch.cuda.synchronize()
        out = u16(runner.out)
        for b, layer, h, ids_, lens_ in pending.pop(step):
            ref = oracle_out(int(ids_[b]), int(lens_[b]), layer, b, h)
            assert_close(out[layer, b, h], ref)

    res = runner.run(reqs, 60, before, after)
    assert not pending
    st, flag = pkv.pkv_check_device_error(runner.err)
    assert st == pkv.PKV_OK and flag == 0
    s = res.stats
    assert s["max_decode_batch"] == max(res.batch_sizes) and s["peak_active"] >= s["max_decode_batch"]
    assert s["allocated_pages"] + s["final_free_pages"] == s["pool_pages"]
    assert res.decode_steps > 0 and res.tokens == sum(res.batch_sizes)
    # admission: under static batching a batch either continues the previous group (its
    # ids a subset: members only finish) or is a whole new group (no id in common);
    # continuous batching admits into a running batch, so some batch mixes the two
    mixed = [bool(a & b) and not b <= a for a, b in zip(batches, batches[1:])]
    if static:
        assert not any(mixed)
        assert sum(1 for a, b in zip(batches, batches[1:]) if not (a & b)) >= 1   # a second group ran
    else:
        assert any(mixed)
    runner.close()
