"""GPU check of DecodeEngine.steps: several decode steps with the micro-batch chains
pipelined across the step boundaries (each chain runs its rows through every step on
its own stream; one join at the end) must write exactly what the same steps write one
by one -- outputs of every step, rotated queries and the pool bytes -- for advancing
positions (each step appends at its own position), BF16 and FP8 pages, and for the
end-to-end form (run_host_steps replaying pipelined graphs).
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300.engine import DecodeEngine
from tests import test_gpu_advance as adv
from tests.test_gpu_parity import dev_bf16, u16

pytestmark = pytest.mark.gpu

STEPS = 9


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def run(c, kv, chains, pipelined, fused=True):
    eng = DecodeEngine(c["num_pages"], c["layers"], c["B"], c["max_blocks"], 2, kv=kv, chains=chains, fused=fused)
    pool0 = torch.from_numpy(c["pool"].view(np.uint8).copy()).cuda()
    eng.slab.copy_(pool0)
    eng.set_tables(c["bt"])
    q = dev_bf16(c["q"][:STEPS])
    k, v = dev_bf16(c["k"][:STEPS]), dev_bf16(c["v"][:STEPS])
    lens = torch.from_numpy(c["lens"][:STEPS]).cuda()
    pos = (lens - 1).contiguous()
    out = torch.zeros_like(q)
    args = [(q[s], k[s], v[s], pos[s], lens[s], out[s]) for s in range(STEPS)]
    eng.step(q[0].clone(), k[0], v[0], pos[0], lens[0], out[0].clone())   # eager: attributes, tensor map
    torch.cuda.synchronize()
    eng.slab.copy_(pool0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if pipelined:
            eng.steps(args)
        else:
            for a in args:
                eng.step(*a)
    g.replay()
    torch.cuda.synchronize()
    st, flag = eng.check_errors()
    res = dict(status=st, flag=flag, out=u16(out), q=u16(q), slab=eng.slab.cpu().numpy())
    eng.close()
    return res


@pytest.mark.parametrize("kv,layers,chains,fused", [("bf16", 2, 3, True), ("bf16", 1, 2, True), ("fp8", 2, 3, True),
                                                    ("bf16", 2, 3, False)])
def test_pipelined_steps_equal_steps_one_by_one(kv, layers, chains, fused):
    c = adv.build_case(kv, layers, seed=120 + layers + (10 if kv == "fp8" else 0))
    one = run(c, kv, chains, pipelined=False, fused=fused)
    pipe = run(c, kv, chains, pipelined=True, fused=fused)
    assert one["status"] == pkv.PKV_OK and pipe["status"] == pkv.PKV_OK and pipe["flag"] == 0
    assert np.array_equal(one["out"], pipe["out"])
    assert np.array_equal(one["q"], pipe["q"])
    assert np.array_equal(one["slab"], pipe["slab"])
    assert np.any(pipe["out"] != 0)


def test_pipelined_end_to_end_graphs():
    from paged_kv_decode_12_gb300 import harness

    outs = {}
    for pipelined in (False, True):
        dw = harness.setup("tiny", pages_per_chunk=1, chains=2)
        io = harness.host_pinned_inputs(dw)
        out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
        bufs = [dw.out] + [torch.empty_like(dw.out) for _ in range(3)]
        dw.eng.run_host_steps(io, bufs, out_host, len(bufs))          # eager pass
        torch.cuda.synchronize()
        graphs = dw.eng.step_graphs(io, bufs, 2, pipelined=pipelined)
        dw.eng.run_host_steps(io, bufs, out_host, 8, graphs=graphs, group=2)
        torch.cuda.synchronize()
        st, flag = dw.eng.check_errors()
        assert st == pkv.PKV_OK and flag == 0
        outs[pipelined] = u16(out_host)
        dw.eng.close()
    assert np.array_equal(outs[False], outs[True])
