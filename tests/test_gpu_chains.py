"""Micro-batch chains of the fused step (DecodeEngine(chains=K)).

The batch rows are cut into K contiguous groups, each a per-layer chain of fused
launches on its own stream, forked from and joined back to the caller's stream.
Sequences never interact, so every output, rotated query and pool byte must be
the same as with one chain, eagerly and inside a CUDA graph, for BF16 and FP8
pages; the chains' workspace counters must be back at zero.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_12_gb300 import harness, launch, pkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def run(name, kv, chains, graph, steps=2):
    cfg = dict(launch.config(name, kv), chains=chains)
    dw = harness.setup(name, **cfg)
    harness.warm(dw, 1)
    dw.reset_q()
    dw.out.zero_()
    if graph:
        cap = harness.capture_steps(dw, steps)
        cap.graph.replay()
    else:
        for _ in range(steps):
            dw.step()
    torch.cuda.synchronize()
    st, flag = dw.eng.check_errors()
    res = dict(status=st, flag=flag, bounds=list(dw.eng.chain_bounds), out=dw.out.cpu().clone(),
               q=dw.q.cpu().clone(), slab=dw.eng.slab.cpu().clone())
    # a call over B rows keeps B x 8 merge counters at the start of its workspace
    ws = dw.eng.chain_ws if chains > 1 else [dw.eng.step_ws]
    rows = np.diff(dw.eng.chain_bounds)
    res["counters_zero"] = all(
        bool((w[: int(n) * 8 * 4].view(torch.int32) == 0).all()) for w, n in zip(ws, rows))
    dw.eng.close()
    return res


def same(a, b):
    return torch.equal(a["out"], b["out"]) and torch.equal(a["q"], b["q"]) and torch.equal(a["slab"], b["slab"])


@pytest.mark.parametrize("graph", [False, True])
def test_tiny_two_chains(graph):
    one = run("tiny", "bf16", 1, graph)
    two = run("tiny", "bf16", 2, graph)
    assert two["bounds"] == [0, 1, 2]
    assert one["status"] == two["status"] == pkv.PKV_OK and two["flag"] == 0
    assert same(one, two) and two["counters_zero"]


def test_b64_chains_bit_identical():
    one = run("b64", "bf16", 1, True)
    assert one["status"] == pkv.PKV_OK and one["counters_zero"]
    for k in (3, launch.CHAINS["b64"]):
        r = run("b64", "bf16", k, True)
        assert len(r["bounds"]) == k + 1 and r["status"] == pkv.PKV_OK and r["flag"] == 0
        assert same(one, r) and r["counters_zero"]


def test_b64_fp8_chains_bit_identical():
    one = run("b64", "fp8", 1, True)
    r = run("b64", "fp8", 3, True)
    assert r["status"] == pkv.PKV_OK and r["flag"] == 0
    assert same(one, r) and r["counters_zero"]
