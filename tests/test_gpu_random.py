"""Randomised GPU parity: seeded draws of batch, lengths, table width, pages per chunk,
ring depth, dispatch order, micro-batch chains, path (one fused launch or the two
named calls) and programmatic dependent launch, each run as one decode step of one
layer and checked against the oracle: every output within the parity tolerance, every
rotated query within one BF16 ulp, and the pool after the step (BF16: placement and
values bit-exact, keys within one ulp; FP8: value codes and scales bit-exact, key rows
within the quantization bound).  Lengths favour page boundaries (16k - 1, 16k, 16k + 1)
and the table is sometimes wider than the longest sequence (empty chunk slots).
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300 import workloads as wl
from paged_kv_decode_12_gb300.engine import DecodeEngine
from tests import paged_helpers as ph
from tests import test_gpu_fp8 as f8
from tests import test_gpu_parity as tp

pytestmark = pytest.mark.gpu

PS = wl.PAGE_SIZE
CHUNKS = [1, 2, 3, 5, 8, 16, 20, 32, 64, 128]


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def draw(seed, kv):
    """One random configuration (a dict) from ``seed``."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 25 if kv == "bf16" else 7))
    top = 2048 if kv == "bf16" else 300
    lens = []
    for _ in range(B):
        r = rng.random()
        if r < 0.4:                      # near a page boundary
            k = int(rng.integers(1, top // PS + 1))
            lens.append(int(np.clip(k * PS + rng.integers(-1, 2), 1, top)))
        elif r < 0.5:
            lens.append(1)
        else:
            lens.append(int(rng.integers(1, top + 1)))
    pages = -(-max(lens) // PS)
    extra = int(rng.integers(0, 9)) if rng.random() < 0.5 else 0
    return dict(lens=lens, max_blocks=min(pages + extra, 128), chunk=int(rng.choice(CHUNKS)),
                ring=int(rng.choice([0, 2, 3, 4])), sorted_units=bool(rng.random() < 0.5),
                chains=int(rng.integers(1, min(B, 3) + 1)), fused=bool(rng.random() < 0.7),
                pdl=bool(rng.random() < 0.8))


def run(c, kv, cfg):
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], cfg["chunk"], kv=kv, fused=cfg["fused"],
                       pdl=cfg["pdl"], ring=cfg["ring"], sorted_units=cfg["sorted_units"], chains=cfg["chains"])
    eng.slab.copy_(torch.from_numpy(c["pool"].view(np.uint8)).cuda())
    eng.set_tables(c["bt"][None])
    lens = torch.from_numpy(c["seq_lens"]).cuda()
    q = tp.dev_bf16(c["q"])[None].contiguous()
    out = torch.full((1, c["B"], 32, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    eng.step(q, tp.dev_bf16(c["k_new"])[None], tp.dev_bf16(c["v_new"])[None], lens - 1, lens, out)
    st, flag = eng.check_errors()
    slab = eng.slab.cpu().numpy()
    res = dict(status=st, flag=flag, out=tp.u16(out)[0], q=tp.u16(q)[0],
               pool=slab.view(np.uint16) if kv == "bf16" else slab)
    eng.close()
    return res


@pytest.mark.parametrize("seed", range(40))
def test_random_bf16_configurations(seed):
    cfg = draw(1000 + seed, "bf16")
    c = tp.make_case(2000 + seed, cfg["lens"], max_blocks=cfg["max_blocks"])
    got = run(c, "bf16", cfg)
    assert got["status"] == pkv.PKV_OK and got["flag"] == 0, cfg
    ref = tp.oracle_run(c)
    tp.assert_close(got["out"], ref["out_f64"])
    assert tp.ulp_distance(got["q"], ref["q"]).max() <= 1, cfg
    assert np.array_equal(np.flatnonzero(got["pool"] != c["pool"]), np.flatnonzero(ref["pool"] != c["pool"])), cfg
    Pg, Pr = ph.pool_view(got["pool"]), ph.pool_view(ref["pool"])
    assert np.array_equal(Pg[:, 1], Pr[:, 1]), cfg
    assert tp.ulp_distance(Pg[:, 0], Pr[:, 0]).max() <= 1, cfg


@pytest.mark.parametrize("seed", range(16))
def test_random_fp8_configurations(seed):
    cfg = draw(3000 + seed, "fp8")
    c = f8.make_case(4000 + seed, cfg["lens"], max_blocks=cfg["max_blocks"])
    got = run(c, "fp8", cfg)
    assert got["status"] == pkv.PKV_OK and got["flag"] == 0, cfg
    ref = f8.oracle_run(c)
    f8.assert_close(got["out"], ref["out_f64"])
    assert tp.ulp_distance(got["q"], ref["q"]).max() <= 1, cfg
    gc, gs = f8.views(got["pool"])
    rc, rs = f8.views(ref["pool"])
    assert np.array_equal(gc[:, 1], rc[:, 1]) and np.array_equal(gs[:, 1].view(np.uint32), rs[:, 1].view(np.uint32))
    written = np.zeros(gc.shape[:1] + gc.shape[2:4], dtype=bool)   # [page][head][slot] of the appended keys
    for b, L in enumerate(c["seq_lens"]):
        written[c["bt"][b, (L - 1) // PS], :, (L - 1) % PS] = True
    assert np.array_equal(gc[:, 0][~written], rc[:, 0][~written])
    assert np.array_equal(gs[:, 0][~written].view(np.uint32), rs[:, 0][~written].view(np.uint32))
    f8.assert_keys_close(gc[:, 0][written], gs[:, 0][written], rc[:, 0][written], rs[:, 0][written])
