"""A bounded wait that runs out, on the GPU, without stalling or faulting anything.

Every wait of the decode kernels on a page copy polls at most a fixed number of
times; a wait that gives up lets the copies still in flight land (bounded), sets
PKV_DEVERR_TIMEOUT in the caller's error flag and lets the kernel finish.  The
option PKV_STEP_TEST_EXPIRE_WAIT makes the first page wait of every work unit of
sequence 0 give up without polling -- the copies it would have waited for are copies
of valid pages, so they land and the drain ends.  The call must return, the flag
must carry the timeout bit (and no other), the merge counters must be back at zero,
every other sequence's outputs must match the oracle, the appends of every sequence
must be in place, and the next call on the same buffers must be correct.
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300.engine import DecodeEngine
from tests import test_gpu_fp8 as f8
from tests import test_gpu_parity as tp

pytestmark = pytest.mark.gpu

LENS = [300, 70, 16, 1, 129, 33]   # sequence 0 spans several 4-page chunks


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def run(c, kv, path, expire, sorted_units=False):
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], 4, kv=kv, fused=path == "fused",
                       sorted_units=sorted_units)
    extra = pkv.PKV_STEP_TEST_EXPIRE_WAIT if expire else 0
    eng.step_options |= extra
    eng.attn_options |= extra
    eng.slab.copy_(torch.from_numpy(c["pool"].view(np.uint8)).cuda())
    eng.set_tables(c["bt"][None])
    q = tp.dev_bf16(c["q"])[None].contiguous()
    lens = torch.from_numpy(c["seq_lens"]).cuda()
    out = torch.full((1, c["B"], 32, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    eng.step(q, tp.dev_bf16(c["k_new"])[None], tp.dev_bf16(c["v_new"])[None], lens - 1, lens, out)
    st, flag = eng.check_errors()
    counters = eng.step_ws[: c["B"] * 8 * 4].view(torch.int32).cpu().numpy()
    slab = eng.slab.cpu().numpy()
    res = dict(status=st, flag=flag, counters=counters, out=tp.u16(out)[0], q=tp.u16(q)[0],
               pool=slab.view(np.uint16) if kv == "bf16" else slab)
    eng.close()
    return res


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("path", ["fused", "separate"])
@pytest.mark.parametrize("sorted_units", [False, True])
def test_expired_wait_flags_timeout_and_the_call_finishes(kv, path, sorted_units):
    c = (f8.make_case if kv == "fp8" else tp.make_case)(90, LENS, max_blocks=32)
    ref = (f8.oracle_run if kv == "fp8" else tp.oracle_run)(c)
    bad = run(c, kv, path, expire=True, sorted_units=sorted_units)
    assert bad["status"] == pkv.PKV_ERR_DEVICE_BOUNDS and bad["flag"] == pkv.PKV_DEVERR_TIMEOUT
    assert np.all(bad["counters"] == 0)
    tp.assert_close(bad["out"][1:], ref["out_f64"][1:])      # every other sequence computed as usual
    assert tp.ulp_distance(bad["q"], ref["q"]).max() <= 1     # every query rotated
    good = run(c, kv, path, expire=False, sorted_units=sorted_units)
    assert good["status"] == pkv.PKV_OK and good["flag"] == 0 and np.all(good["counters"] == 0)
    tp.assert_close(good["out"], ref["out_f64"])
    # the appends (sequence 0's included) happened before any wait: same pool bytes
    assert np.array_equal(bad["pool"], good["pool"])


def test_expire_option_is_rejected_by_the_two_kernel_form():
    c = tp.make_case(91, [20, 40])
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], 1, fused=False, split_merge=True)
    eng.set_tables(c["bt"][None])
    q = tp.dev_bf16(c["q"])
    out = torch.zeros_like(q)
    lens = torch.from_numpy(c["seq_lens"]).cuda()
    with pytest.raises(pkv.PkvError) as e:
        eng.attention(0, q, lens, out, variant=pkv.PKV_DECODE_SPLIT_MERGE | pkv.PKV_STEP_TEST_EXPIRE_WAIT)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    eng.close()
