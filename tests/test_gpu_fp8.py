"""GPU parity of the FP8 KV pages (through the C ABI) against the FP64 oracle.

The scheme ("从零构建大模型推理引擎：KV缓存、算子融合与量化优化实战", section 5.1,
read as E4M3 codes with one FP32 amax/448 scale per (token, KV head) row) is the
oracle's; these tests hold the CUDA path to it:
  * placement: exactly the appended rows' bytes change;
  * V codes and scales: bit-exact (same BF16 input, same FP32 arithmetic);
  * K: the rotated key can differ from the oracle's by one BF16 ulp, so codes may
    differ by one step where that ulp crosses a rounding boundary; the test bounds
    the dequantized difference and requires almost all codes to be equal;
  * attention over FP8 pages: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|, the oracle
    dequantizing in FP64;
  * the step entry point equals the separate calls bit for bit, device checks set
    the flag instead of faulting, and the bench's launch configuration agrees
    with the oracle on sampled units at full size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_12_gb300 import harness, launch, pkv
from paged_kv_decode_12_gb300 import workloads as wl
from paged_kv_decode_12_gb300.engine import DecodeEngine
from tests import paged_helpers as ph

pytestmark = pytest.mark.gpu

HQ, HKV, D, PS = wl.NUM_Q_HEADS, wl.NUM_KV_HEADS, wl.HEAD_DIM, wl.PAGE_SIZE
PAGE = oracle.FP8_PAGE_BYTES
CODES = 2 * HKV * PS * D
SCALE = 1.0 / math.sqrt(D)
ATOL = RTOL = 1e-2
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16).cuda()


def views(pool: np.ndarray):
    """(codes [pages][2][8][16][64] (a copy, through the oracle's byte layout), scales
    [pages][2][8][16] (a view)) of an FP8 pool."""
    pv = ph.Fp8Pages(pool)
    return pv.codes(), pv.scales


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def key(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)

    return np.abs(key(a) - key(b))


def make_case(seed, seq_lens, num_pages=None, max_blocks=None):
    """Cached tokens 0..L-2 quantized by the oracle into a sentinel-filled FP8 pool;
    token L-1 is the one appended by the step."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B, S = seq_lens.size, int(seq_lens.max())
    max_blocks = max_blocks or -(-S // PS)
    num_pages = num_pages or ph.pages_needed(seq_lens) + 2
    bt = wl.permutation_block_tables(rng, seq_lens, num_pages, max_blocks)
    pool = np.full(num_pages * PAGE, SENTINEL, dtype=np.uint8)
    pv = ph.Fp8Pages(pool)
    for b, L in enumerate(seq_lens):
        for t in range(int(L) - 1):
            page, slot = bt[b, t // PS], t % PS
            for kv in (0, 1):
                for h in range(HKV):
                    pv.set_row(page, kv, h, slot, *oracle.quantize_row_fp8(wl.bf16_normal_host(rng, (D,))))
    q = wl.bf16_normal_host(rng, (B, HQ, D))
    k_new = wl.bf16_normal_host(rng, (B, HKV, D))
    v_new = wl.bf16_normal_host(rng, (B, HKV, D))
    return dict(seq_lens=seq_lens, B=B, max_blocks=max_blocks, num_pages=num_pages, q=q, k_new=k_new,
                v_new=v_new, bt=bt, pool=pool)


def engine_for(c, chunk=16, fused=False):
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], chunk, kv="fp8", fused=fused)
    eng.slab.copy_(torch.from_numpy(c["pool"]).cuda())
    eng.set_tables(c["bt"][None])
    return eng


def gpu_run(c, chunk=16, append=True, seq_lens_override=None):
    eng = engine_for(c, chunk)
    q = dev_bf16(c["q"])
    lens = c["seq_lens"] if seq_lens_override is None else np.asarray(seq_lens_override, np.int32)
    lens_d = torch.from_numpy(lens).cuda()
    pos_d = torch.from_numpy(c["seq_lens"] - 1).cuda()
    out = torch.full((c["B"], HQ, D), 7.0, dtype=torch.bfloat16, device="cuda")
    if append:
        eng.append(0, dev_bf16(c["k_new"]), dev_bf16(c["v_new"]), q, pos_d)
    eng.attention(0, q, lens_d, out)
    status, flag = eng.check_errors()
    res = dict(pool=eng.slab.cpu().numpy(), q=u16(q), out=u16(out), status=status, flag=flag)
    eng.close()
    return res


def oracle_run(c, append=True):
    pool = c["pool"].copy()
    q = c["q"].copy()
    g = oracle.geom(c["num_pages"])
    if append:
        oracle.append_fp8(pool, g, c["bt"], c["seq_lens"] - 1, c["k_new"], c["v_new"], q)
    out_bf16, out_f64 = oracle.decode_fp8(pool, g, c["bt"], c["seq_lens"], q, SCALE)
    return dict(pool=pool, q=q, out=out_bf16, out_f64=out_f64)


def assert_close(gpu_u16, ref_f64):
    got = ph.bf16_to_f64(gpu_u16)
    err = np.abs(got - ref_f64)
    bound = ATOL + RTOL * np.abs(ref_f64)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"max excess at {worst}: got {got[worst]} ref {ref_f64[worst]}"


def assert_keys_close(gpu_codes, gpu_scales, ref_codes, ref_scales):
    """K rows quantized from keys that may differ by one BF16 ulp."""
    assert np.all(np.abs(gpu_scales / ref_scales - 1) <= 2.0**-7)
    xg = oracle.e4m3_to_f64(gpu_codes) * gpu_scales[..., None].astype(np.float64)
    xr = oracle.e4m3_to_f64(ref_codes) * ref_scales[..., None].astype(np.float64)
    # two half-steps of E4M3 (2^-4 relative each), one BF16 ulp, the subnormal half-steps
    bound = (2.0**-3 + 2.0**-7) * np.abs(xr) + 2.0**-9 * ref_scales[..., None]
    assert np.all(np.abs(xg - xr) <= bound * (1 + 1e-9))
    assert np.mean(gpu_codes == ref_codes) >= 0.95


# ---------------------------------------------------------------------------- append

@pytest.mark.parametrize("seq_lens", [[1], [16, 17, 33], [2, 31, 100, 64, 65]])
def test_fp8_append_placement_and_codes(seq_lens):
    c = make_case(11, seq_lens)
    gpu, ref = gpu_run(c), oracle_run(c)
    assert gpu["status"] == pkv.PKV_OK and gpu["flag"] == 0
    gc, gs = views(gpu["pool"])
    rc, rs = views(ref["pool"])
    # every byte outside the appended K rows is the oracle's (placement + V bit-exact)
    krows = np.zeros(gc.shape[:4], dtype=bool)
    for b, L in enumerate(c["seq_lens"]):
        krows[c["bt"][b, (L - 1) // PS], 0, :, (L - 1) % PS] = True
    assert np.array_equal(gc[~krows], rc[~krows])
    assert np.array_equal(gs[~krows].view(np.uint32), rs[~krows].view(np.uint32))
    changed = np.count_nonzero(ref["pool"] != c["pool"])
    assert changed <= len(seq_lens) * 2 * HKV * (D + 4)
    assert_keys_close(gc[krows], gs[krows], rc[krows], rs[krows])
    # queries rotated as on the BF16 path: within one BF16 ulp
    assert ulp_distance(gpu["q"], ref["q"]).max() <= 1


def test_fp8_prefill_matches_oracle_appends():
    rng = np.random.default_rng(5)
    layers, T, start = 2, 37, 3
    max_blocks = 4
    num_pages = 2 * max_blocks + 1
    # layers never share pages (as pkv_block_tables_build guarantees)
    bt_rows = rng.permutation(num_pages)[:layers * max_blocks].reshape(layers, max_blocks).astype(np.int32)
    k = wl.bf16_normal_host(rng, (layers, T, HKV, D))
    v = wl.bf16_normal_host(rng, (layers, T, HKV, D))
    eng = DecodeEngine(num_pages, layers, 1, max_blocks, 4, kv="fp8")
    eng.slab.fill_(SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_prefill_append(eng.pool, dev_bf16(k), dev_bf16(v), torch.from_numpy(bt_rows).cuda(), max_blocks, layers,
                           start, T, eng.rope, eng.max_pos, err)
    st, flag = pkv.pkv_check_device_error(err)
    assert st == pkv.PKV_OK and flag == 0
    got = eng.slab.cpu().numpy()
    eng.close()
    ref = np.full(num_pages * PAGE, SENTINEL, dtype=np.uint8)
    g = oracle.geom(num_pages)
    for l in range(layers):
        for t in range(T):
            oracle.append_fp8(ref, g, bt_rows[l][None], [start + t], k[l, t][None], v[l, t][None])
    gc, gs = views(got)
    rc, rs = views(ref)
    assert np.array_equal(gc[:, 1], rc[:, 1]) and np.array_equal(gs[:, 1].view(np.uint32), rs[:, 1].view(np.uint32))
    written = np.zeros(gc.shape[:4], dtype=bool)
    for l in range(layers):
        for t in range(T):
            p = start + t
            written[bt_rows[l, p // PS], 0, :, p % PS] = True
    assert np.array_equal(gc[~written], rc[~written])
    assert_keys_close(gc[written], gs[written], rc[written], rs[written])


# ---------------------------------------------------------------------------- attention

@pytest.mark.parametrize("chunk", [1, 3, 16, 128])
def test_fp8_attention_parity_ragged(chunk):
    c = make_case(21, [2, 3, 16, 17, 18, 32, 34, 65, 101, 201])
    # attention over the L-1 cached tokens (the slot of token L-1 holds sentinel bytes)
    c = dict(c, seq_lens=c["seq_lens"] - 1)
    gpu = gpu_run(c, chunk=chunk, append=False)
    ref = oracle_run(c, append=False)
    assert gpu["status"] == pkv.PKV_OK and gpu["flag"] == 0
    assert_close(gpu["out"], ref["out_f64"])


@pytest.mark.parametrize("chunk", [2, 16])
def test_fp8_append_then_attention_parity(chunk):
    c = make_case(31, [1, 16, 17, 48, 129])
    gpu, ref = gpu_run(c, chunk=chunk), oracle_run(c)
    assert gpu["status"] == pkv.PKV_OK and gpu["flag"] == 0
    assert_close(gpu["out"], ref["out_f64"])


def test_fp8_single_token_returns_dequantized_v():
    c = make_case(41, [1, 1, 1])
    gpu, ref = gpu_run(c), oracle_run(c)
    assert ulp_distance(gpu["out"], ref["out"]).max() <= 1


def fp8_step_run(c, chunk, fused, ring=0, sorted_units=False, pdl=True, repeats=1, lens_override=None):
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], chunk, kv="fp8", fused=fused, ring=ring,
                       sorted_units=sorted_units, pdl=pdl)
    eng.slab.copy_(torch.from_numpy(c["pool"]).cuda())
    eng.set_tables(c["bt"][None])
    lens = c["seq_lens"] if lens_override is None else np.asarray(lens_override, np.int32)
    lens_d = torch.from_numpy(lens).cuda()
    for _ in range(repeats):
        q = dev_bf16(c["q"])[None].contiguous()
        out = torch.zeros((1, c["B"], HQ, D), dtype=torch.bfloat16, device="cuda")
        eng.step(q, dev_bf16(c["k_new"])[None], dev_bf16(c["v_new"])[None], lens_d - 1, lens_d, out)
    st, flag = eng.check_errors()
    counters = eng.step_ws[: c["B"] * 8 * 4].view(torch.int32).cpu().numpy()
    res = dict(out=u16(out)[0], q=u16(q)[0], pool=eng.slab.cpu().numpy(), status=st, flag=flag, counters=counters)
    eng.close()
    return res


@pytest.mark.parametrize("chunk", [1, 4, 128])
@pytest.mark.parametrize("ring,sorted_units", [(0, False), (2, False), (3, True)])
def test_fp8_fused_step_equals_separate_calls(chunk, ring, sorted_units):
    # one launch per layer (append + quantize + attention + merge) against the
    # quantizing append and the FP8 split kernel: same pool bytes, queries, outputs
    c = make_case(51, [5, 16, 17, 77, 130, 1, 200, 33])
    sep = fp8_step_run(c, chunk, fused=False)
    fus = fp8_step_run(c, chunk, fused=True, ring=ring, sorted_units=sorted_units, repeats=1)
    assert sep["status"] == pkv.PKV_OK and fus["status"] == pkv.PKV_OK and fus["flag"] == 0
    assert np.all(fus["counters"] == 0)
    assert np.array_equal(sep["out"], fus["out"]) and np.array_equal(sep["pool"], fus["pool"])
    assert np.array_equal(sep["q"], fus["q"])
    assert_close(fus["out"], oracle_run(c)["out_f64"])


def test_fp8_fused_step_repeats_and_without_pdl():
    c = make_case(52, [40, 3, 129])
    a = fp8_step_run(c, 2, fused=True)
    b = fp8_step_run(c, 2, fused=True, pdl=False)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["pool"], b["pool"])
    r = fp8_step_run(c, 2, fused=True, repeats=3)   # the counters stay usable across calls
    assert r["status"] == pkv.PKV_OK and np.all(r["counters"] == 0)


def test_fp8_fused_step_device_checks():
    c = make_case(53, [40, 20, 70])
    z = fp8_step_run(c, 4, fused=True, lens_override=[40, 0, 70])
    assert z["flag"] & pkv.PKV_DEVERR_LENGTH and np.all(z["out"][1] == 0) and np.all(z["counters"] == 0)
    ref = fp8_step_run(c, 4, fused=False)
    assert np.array_equal(z["out"][[0, 2]], ref["out"][[0, 2]])
    bad = dict(c, bt=c["bt"].copy())
    bad["bt"][2, 1] = c["num_pages"] + 3
    f = fp8_step_run(bad, 4, fused=True)
    assert f["flag"] & pkv.PKV_DEVERR_PAGE_RANGE and np.all(f["counters"] == 0)
    assert np.array_equal(f["out"][:2], ref["out"][:2])


def test_fp8_bad_page_id_sets_flag():
    c = make_case(61, [40, 20])
    c["bt"][1, 0] = c["num_pages"] + 5
    gpu = gpu_run(c, append=False)
    assert gpu["status"] == pkv.PKV_ERR_DEVICE_BOUNDS and gpu["flag"] & pkv.PKV_DEVERR_PAGE_RANGE
    assert np.all(gpu["out"][1] == 0)
    # the other sequence is unaffected
    ok = dict(c, seq_lens=c["seq_lens"][:1], bt=c["bt"][:1], q=c["q"][:1], B=1)
    assert_close(gpu["out"][0], oracle_run(ok, append=False)["out_f64"][0])


def test_fp8_zero_length_sets_flag_and_zeros():
    c = make_case(71, [10, 30])
    gpu = gpu_run(c, append=False, seq_lens_override=[0, 29])
    assert gpu["flag"] & pkv.PKV_DEVERR_LENGTH
    assert np.all(gpu["out"][0] == 0)


# ---------------------------------------------------------------------------- full size, bench configuration

@pytest.mark.parametrize("name,layers", [("b64", tuple(range(16))), ("b256", (0, 15))])
def test_fp8_full_size_every_unit(name, layers):
    # every (layer, sequence, query head) of a whole b64 step and of two whole b256 layers
    # over FP8 pages, at the benchmark's launch settings, against the FP8 oracle
    from tests import full_size

    checked = full_size.check_full_size(name, "fp8", layers)
    assert checked == wl.make_workload(name).batch * len(layers) * HQ
