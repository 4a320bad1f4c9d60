"""GPU parity of the fused per-layer step (pkv_decode_step).

The fused kernel must produce bit-for-bit what pkv_append_rope (at seq_len - 1)
followed by pkv_decode_attention produce -- the same pool bytes, the same rotated
queries, the same outputs -- for both compute policies and every chunk size; and
therefore match the oracle within the parity tolerance.  Its per-(sequence, KV
head) counters must be back at zero after every call, and launching with or
without programmatic dependent launch must not change a bit.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300.engine import DecodeEngine
from tests.test_gpu_parity import RAGGED, VARIANTS, assert_close, dev_bf16, gpu_run, make_case, oracle_run, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


# "sorted": units dispatched largest first (PKV_STEP_SORTED); "grid": in grid order
SCHEDULES = ["grid", "sorted"]


def fused_run(c, chunk=16, variant=pkv.PKV_DECODE_DEFAULT, pdl=True, seq_lens_override=None, repeats=1,
              schedule="auto", ring=0):
    sorted_units = schedule == "sorted"
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], chunk, variant, pdl=pdl, ring=ring,
                       sorted_units=sorted_units)
    eng.slab.copy_(torch.from_numpy(c["pool"].view(np.uint8)).cuda())
    eng.set_tables(c["bt"][None])
    lens = c["seq_lens"] if seq_lens_override is None else np.asarray(seq_lens_override, np.int32)
    lens_d = torch.from_numpy(lens).cuda()
    k_new, v_new = dev_bf16(c["k_new"]), dev_bf16(c["v_new"])
    outs = []
    for _ in range(repeats):
        q = dev_bf16(c["q"])
        out = torch.full((c["B"], 32, 64), 7.0, dtype=torch.bfloat16, device="cuda")
        eng.fused_layer(0, q, k_new, v_new, lens_d, out)
        outs.append(u16(out))
    status, flag = eng.check_errors()
    counters = eng.step_ws[: c["B"] * 8 * 4].view(torch.int32).cpu().numpy()
    res = dict(pool=u16(eng.slab.view(torch.bfloat16)), q=u16(q), out=outs[-1], outs=outs, status=status,
               flag=flag, counters=counters)
    eng.close()
    return res


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("chunk", [1, 3, 16, 128])
def test_fused_is_bit_identical_to_separate_calls(schedule, variant, chunk):
    c = make_case(31, RAGGED, max_blocks=128)
    f = fused_run(c, chunk=chunk, variant=variant, schedule=schedule)
    s = gpu_run(c, chunk=chunk, variant=variant)
    assert f["status"] == pkv.PKV_OK and f["flag"] == 0
    assert np.array_equal(f["pool"], s["pool"])
    assert np.array_equal(f["q"], s["q"])
    assert np.array_equal(f["out"], s["out"])
    assert np.all(f["counters"] == 0)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("variant", VARIANTS)
def test_fused_tiny_vs_oracle(schedule, variant):
    c = make_case(12, [17, 40], num_pages=8)
    f, o = fused_run(c, variant=variant, schedule=schedule), oracle_run(c)
    assert_close(f["out"], o["out_f64"])


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_fused_repeated_calls_and_pdl_switch(schedule):
    c = make_case(32, [2048, 600, 1, 17, 999], max_blocks=128)
    a = fused_run(c, chunk=8, repeats=3, schedule=schedule)
    b = fused_run(c, chunk=8, pdl=False, schedule=schedule)
    assert all(np.array_equal(o, a["outs"][0]) for o in a["outs"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["pool"], b["pool"])
    assert np.all(a["counters"] == 0) and np.all(b["counters"] == 0)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("variant", VARIANTS)
def test_fused_bad_page_sets_flag_and_resets_counters(schedule, variant):
    c = make_case(33, [300, 200, 64], max_blocks=32)
    bad = c["bt"].copy()
    bad[0, 3] = c["num_pages"] + 5
    f = fused_run(dict(c, bt=bad), chunk=4, variant=variant, schedule=schedule)
    assert f["status"] == pkv.PKV_ERR_DEVICE_BOUNDS and f["flag"] & pkv.PKV_DEVERR_PAGE_RANGE
    assert np.all(f["counters"] == 0)
    o = oracle_run(c)
    assert_close(f["out"][1:], o["out_f64"][1:])          # untouched sequences stay right


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_fused_zero_length_sets_flag_and_zeros(schedule):
    c = make_case(34, [20, 30])
    f = fused_run(c, seq_lens_override=[0, 30], schedule=schedule)
    assert f["flag"] & pkv.PKV_DEVERR_LENGTH
    assert np.all(f["out"][0] == 0)
    assert_close(f["out"][1], oracle_run(c)["out_f64"][1])


@pytest.mark.parametrize("ring", [2, 3])
def test_ring_depth_changes_no_bit(ring):
    c = make_case(36, RAGGED, max_blocks=128)
    a = fused_run(c, chunk=8)
    b = fused_run(c, chunk=8, ring=ring)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["pool"], b["pool"])
    assert np.array_equal(a["q"], b["q"]) and np.all(b["counters"] == 0)


def test_sorted_many_units_per_launch():
    # far more units than resident CTAs (batch 300, 2-page chunks): several waves, the
    # sorted order covering every unit exactly once
    rng = np.random.default_rng(35)
    lens = rng.integers(1, 300, size=300)
    c = make_case(35, lens, max_blocks=64)
    g = fused_run(c, chunk=2, schedule="grid")
    p = fused_run(c, chunk=2, schedule="sorted", repeats=2)
    assert p["status"] == pkv.PKV_OK and np.all(p["counters"] == 0)
    assert np.array_equal(p["out"], g["out"]) and np.array_equal(p["pool"], g["pool"])
    assert np.array_equal(p["q"], g["q"])


@pytest.mark.parametrize("chunk", [1, 5, 32])
def test_sorted_order_with_invalid_lengths_and_ring(chunk):
    # every unit size class (full chunks, several last-chunk sizes, an invalid length
    # at both ends) in one launch; the sorted order must still cover each unit once
    rng = np.random.default_rng(37)
    lens = np.concatenate([[2048, 1, 16, 17], rng.integers(1, 2048, size=60)]).astype(np.int32)
    c = make_case(37, lens, max_blocks=128)
    g = fused_run(c, chunk=chunk, schedule="grid")
    for ring, sched in ((0, "sorted"), (2, "sorted"), (3, "sorted")):
        s_ = fused_run(c, chunk=chunk, schedule=sched, ring=ring, repeats=2)
        assert s_["status"] == pkv.PKV_OK and np.all(s_["counters"] == 0)
        assert np.array_equal(s_["out"], g["out"]) and np.array_equal(s_["pool"], g["pool"])
        assert np.array_equal(s_["q"], g["q"])
    bad = fused_run(c, chunk=chunk, schedule="sorted", seq_lens_override=np.where(np.arange(lens.size) % 7 == 3, 0,
                                                                                    lens))
    assert bad["flag"] & pkv.PKV_DEVERR_LENGTH and np.all(bad["counters"] == 0)
    zero = np.arange(lens.size) % 7 == 3
    assert np.all(bad["out"][zero] == 0)
    assert np.array_equal(bad["out"][~zero], g["out"][~zero])


def test_run_host_equals_device_step():
    # the end-to-end form (packed pinned inputs, one copy each way) computes the same step
    from paged_kv_decode_12_gb300 import harness

    dw = harness.setup("tiny", pages_per_chunk=1, ring=2)
    pool0 = dw.eng.slab.clone()
    dw.step()
    torch.cuda.synchronize()
    ref = u16(dw.out)
    dw.eng.slab.copy_(pool0)
    io = harness.host_pinned_inputs(dw)
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    dw.eng.run_host(io, dw.out, out_host)
    torch.cuda.synchronize()
    assert np.array_equal(u16(out_host), ref)
    assert io.bytes == sum(t.numel() * t.element_size() for t in (dw.q0, dw.k_new, dw.v_new, dw.pos, dw.seq_lens))
    dw.eng.close()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_step_layers_call_matches_per_layer_calls(kv):
    # pkv_decode_step_layers (one call for every layer, the engine's step) against one
    # pkv_decode_step call per layer on the same inputs: every byte equal
    from paged_kv_decode_12_gb300 import harness

    res = []
    for per_layer in (False, True):
        dw = harness.setup("b8", layers=4, pages_per_chunk=16, ring=2, kv=kv)
        dw.reset_q()
        if per_layer:
            for layer in range(dw.w.layers):
                dw.eng.fused_layer(layer, dw.q[layer], dw.k_new[layer], dw.v_new[layer], dw.seq_lens, dw.out[layer])
        else:
            dw.step()
        torch.cuda.synchronize()
        st, flag = dw.eng.check_errors()
        assert st == pkv.PKV_OK and flag == 0
        res.append((dw.out.cpu().clone(), dw.q.cpu().clone(), dw.eng.slab.cpu().clone()))
        dw.eng.close()
    for a, b in zip(*res):
        assert torch.equal(a, b)


@pytest.mark.parametrize("chains,buffers", [(1, 2), (2, 2), (2, 3), (1, 4)])
def test_run_host_steps_rotating_buffers(chains, buffers):
    # the end-to-end steps through rotating buffers compute what the plain step computes:
    # every step's output reaches the host, and the last one stays there
    from paged_kv_decode_12_gb300 import harness

    dw = harness.setup("tiny", pages_per_chunk=1, ring=2, chains=chains)
    pool0 = dw.eng.slab.clone()
    dw.step()
    torch.cuda.synchronize()
    ref = u16(dw.out)
    io = harness.host_pinned_inputs(dw)
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    outs = [dw.out] + [torch.empty_like(dw.out) for _ in range(buffers - 1)]
    for steps in (1, 2, 5):
        dw.eng.slab.copy_(pool0)
        out_host.zero_()
        for o in outs:
            o.zero_()
        dw.eng.run_host_steps(io, outs, out_host, steps)
        torch.cuda.synchronize()
        assert np.array_equal(u16(out_host), ref), steps
        for o in outs[:steps]:
            assert np.array_equal(u16(o), ref), steps
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dw.eng.run_host_steps(io, outs, out_host, 3)
    dw.eng.slab.copy_(pool0)
    out_host.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(u16(out_host), ref)
    # the same steps with the kernels replayed from graphs of `group` steps, copies between
    for group in (1, 2):
        if len(outs) % group:
            continue
        graphs = dw.eng.step_graphs(io, outs, group)
        for steps in (group, len(outs) + 2 * group):
            dw.eng.slab.copy_(pool0)
            out_host.zero_()
            for o in outs:
                o.zero_()
            dw.eng.run_host_steps(io, outs, out_host, steps, graphs=graphs, group=group)
            torch.cuda.synchronize()
            assert np.array_equal(u16(out_host), ref), (group, steps)
            for o in outs[:steps]:
                assert np.array_equal(u16(o), ref), (group, steps)
    st, flag = dw.eng.check_errors()
    assert st == pkv.PKV_OK and flag == 0
    dw.eng.close()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("chunk", [16, 20, 43, 64])   # 8, 7, 3 and 2 chunk slots at 128 table entries
def test_in_kernel_merge_equals_two_kernel_form(kv, chunk):
    # the fused step and the default attention call merge chunk partials inside the launch
    # (ticket); the two-kernel form merges them in a second kernel: same bits
    from tests import test_gpu_fp8 as f8

    lens = [2048, 1, 16, 17, 320, 321, 1000, 640, 641, 1500, 33, 2047]
    c = (f8.make_case if kv == "fp8" else make_case)(38, lens, max_blocks=128)
    pool = c["pool"].view(np.uint8)

    def run(fused, split_merge):
        eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], chunk, kv=kv, fused=fused,
                           split_merge=split_merge)
        eng.slab.copy_(torch.from_numpy(pool).cuda())
        eng.set_tables(c["bt"][None])
        lens_d = torch.from_numpy(c["seq_lens"]).cuda()
        outs = []
        for _ in range(2):   # a second call on the same workspace
            q = dev_bf16(c["q"])[None].contiguous()
            out = torch.full((1, c["B"], 32, 64), 7.0, dtype=torch.bfloat16, device="cuda")
            eng.step(q, dev_bf16(c["k_new"])[None], dev_bf16(c["v_new"])[None], lens_d - 1, lens_d, out)
            outs.append(u16(out)[0])
        st, flag = eng.check_errors()
        counters = eng.step_ws[: c["B"] * 8 * 4].view(torch.int32).cpu().numpy()
        res = dict(out=outs, q=u16(q)[0], pool=eng.slab.cpu().numpy(), st=st, flag=flag, counters=counters)
        eng.close()
        return res

    fused = run(True, False)
    sep = run(False, False)
    two_kernel = run(False, True)
    for r in (fused, sep, two_kernel):
        assert r["st"] == pkv.PKV_OK and r["flag"] == 0 and np.all(r["counters"] == 0)
        assert np.array_equal(r["out"][0], r["out"][1])
    for r in (sep, two_kernel):
        assert np.array_equal(fused["out"][0], r["out"][0])
        assert np.array_equal(fused["pool"], r["pool"])
    ref = (f8.oracle_run if kv == "fp8" else oracle_run)(c)
    assert_close(fused["out"][0], ref["out_f64"])
