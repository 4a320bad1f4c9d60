"""The no-allocation decode entry point (GPU).

``pkv_decode_attention_noalloc`` serves callers that cannot allocate device
memory -- a plugin inside an engine that owns the whole device-memory budget, a
loop that must not call cudaMalloc/cudaFree because they can synchronise the
device, a C caller without a device allocator.  It keeps the chunk partials in
the library's static device scratch instead of a caller workspace.  This test
calls it through the C ABI twice in a row, on different inputs (so the second
call runs over the first call's leftovers in the shared scratch), and checks each
result against the regular ``pkv_decode_attention`` on the same inputs, within
the tolerance the parity tests use.  It also checks the size limit.  The file is
named so that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

from paged_kv_decode_12_gb300 import pkv
from paged_kv_decode_12_gb300 import workloads as wl
from paged_kv_decode_12_gb300.engine import DecodeEngine

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2
SCALE = 1.0 / math.sqrt(wl.HEAD_DIM)


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def _bf16(t):
    return t.float().cpu().numpy().astype(np.float64)


def _inputs(seed, seq_lens, max_blocks=128, kv="bf16", pages_per_chunk=16):
    lens = np.asarray(seq_lens, dtype=np.int32)
    B = lens.size
    need = int(sum(-(-int(L) // wl.PAGE_SIZE) for L in lens))
    eng = DecodeEngine(need + 4, 1, B, max_blocks, pages_per_chunk=pages_per_chunk, kv=kv)
    if kv == "fp8":
        codes, scales = eng.fp8_views()
        wl.fill_fp8_pages_(codes, scales, seed, 0.0)
    else:
        wl.fill_bf16_normal_(eng.pool_view(), seed)
    eng.build_tables(lens)
    q = wl.fill_bf16_normal_(torch.empty((B, wl.NUM_Q_HEADS, wl.HEAD_DIM), dtype=torch.bfloat16, device="cuda"),
                             seed + 1)
    return eng, q, torch.from_numpy(lens).cuda()


def _regular(eng, q, lens):
    out = torch.zeros_like(q)
    eng.attention(0, q, lens, out)
    return out


def _noalloc(eng, q, lens):
    out = torch.full_like(q, 3.0)
    pkv.pkv_decode_attention_noalloc(eng.pool, q, eng.bt[0], eng.max_blocks, lens, eng.batch, eng.scale,
                                     eng.pages_per_chunk, out, eng.err)
    return out


def test_noalloc_matches_regular_on_two_calls_in_a_row():
    cases = [(21, [2048, 700, 33, 1, 1500, 16, 17, 257]),   # several chunks per sequence
             (22, [40, 2048, 5, 300])]                      # fewer chunks: leftovers stay in the scratch
    for seed, lens in cases:
        eng, q, lens_d = _inputs(seed, lens)
        ref = _bf16(_regular(eng, q, lens_d))
        got = _bf16(_noalloc(eng, q, lens_d))
        torch.cuda.synchronize()
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
        st, flag = eng.check_errors()
        assert st == pkv.PKV_OK and flag == 0
        eng.close()


def test_noalloc_fp8_pool_matches_regular():
    # FP8 pages: the split kernel keeps its chunk partials in the static scratch too
    for seed, lens in [(24, [2048, 90, 1, 513]), (25, [17, 640])]:
        eng, q, lens_d = _inputs(seed, lens, kv="fp8")
        ref = _bf16(_regular(eng, q, lens_d))
        got = _bf16(_noalloc(eng, q, lens_d))
        torch.cuda.synchronize()
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
        st, flag = eng.check_errors()
        assert st == pkv.PKV_OK and flag == 0
        eng.close()


def test_noalloc_single_chunk_after_multi_chunk():
    # a call whose sequences all fit one chunk writes its outputs directly (no partials,
    # no merge) -- after a multi-chunk call has left partials in the scratch
    eng, q, lens_d = _inputs(26, [2048, 1000, 37])
    first, ref = _bf16(_noalloc(eng, q, lens_d)), _bf16(_regular(eng, q, lens_d))
    torch.cuda.synchronize()
    assert np.all(np.abs(first - ref) <= ATOL + RTOL * np.abs(ref))
    eng.close()
    eng, q, lens_d = _inputs(27, [5, 16, 17, 40], max_blocks=4, pages_per_chunk=4)
    ref = _bf16(_regular(eng, q, lens_d))
    got = _bf16(_noalloc(eng, q, lens_d))
    torch.cuda.synchronize()
    assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    st, flag = eng.check_errors()
    assert st == pkv.PKV_OK and flag == 0
    eng.close()


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    eng, q, lens_d = _inputs(23, [64, 64])
    B_too_big = 4096                       # 4096 x 32 heads x 8 chunks x 264 B > 32 MiB
    assert pkv.pkv_decode_workspace_bytes(B_too_big, 128, 16) > pkv.PKV_NOALLOC_SCRATCH_BYTES
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_noalloc(eng.pool, q, eng.bt[0], 128, lens_d, B_too_big, SCALE, 16, q, eng.err)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE_TOO_SMALL
    eng.close()
