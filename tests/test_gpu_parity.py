"""GPU parity: libpkv's kernels (through the C ABI) against the FP64 CPU oracle.

Bars (from the engine's statement of the problem):
  * page / slot addressing and append placement: bit-exact (sentinel-filled pool:
    exactly the oracle's bytes change, V bit-identical);
  * appended RoPE'd keys and rotated queries: within 1 BF16 ulp of the oracle;
  * attention outputs: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| (oracle in FP64);
  * L = 1 returns v exactly; physical page order and batch composition change
    no bit; one chunk vs one page per chunk agree to FP32 rounding;
  * device-side bounds checks set the error flag instead of faulting.
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
SCALE = 1.0 / math.sqrt(D)
ATOL = RTOL = 1e-2
VARIANTS = [pkv.PKV_DECODE_SIMT, pkv.PKV_DECODE_MMA]


@pytest.fixture(scope="module", autouse=True)
def native():
    from paged_kv_decode_12_gb300 import _build

    _build.build()
    pkv.lib()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16).cuda()


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def key(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)

    return np.abs(key(a) - key(b))


def make_case(seed, seq_lens, num_pages=None, max_blocks=None, perm_seed=None):
    """Cached tokens 0..L-2 scattered into a sentinel-filled pool; token L-1 is appended."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B, S = seq_lens.size, int(seq_lens.max())
    max_blocks = max_blocks or -(-S // PS)
    num_pages = num_pages or ph.pages_needed(seq_lens) + 2
    K = wl.bf16_normal_host(rng, (B, HKV, S, D))
    V = wl.bf16_normal_host(rng, (B, HKV, S, D))
    q = wl.bf16_normal_host(rng, (B, HQ, D))
    k_new = wl.bf16_normal_host(rng, (B, HKV, D))
    v_new = wl.bf16_normal_host(rng, (B, HKV, D))
    prng = np.random.default_rng(perm_seed) if perm_seed is not None else rng
    bt = wl.permutation_block_tables(prng, seq_lens, num_pages, max_blocks)
    pool = ph.scatter_tokens(ph.new_pool(num_pages), bt, seq_lens - 1, K, V)
    return dict(seq_lens=seq_lens, B=B, max_blocks=max_blocks, num_pages=num_pages, K=K, V=V, q=q,
                k_new=k_new, v_new=v_new, bt=bt, pool=pool)


def gpu_run(c, chunk=16, variant=pkv.PKV_DECODE_DEFAULT, append=True, seq_lens_override=None, pos_override=None):
    eng = DecodeEngine(c["num_pages"], 1, c["B"], c["max_blocks"], chunk, variant)
    eng.slab.copy_(torch.from_numpy(c["pool"].view(np.uint8)).cuda())
    eng.set_tables(c["bt"][None])
    q = dev_bf16(c["q"])
    lens = c["seq_lens"] if seq_lens_override is None else np.asarray(seq_lens_override, np.int32)
    pos = c["seq_lens"] - 1 if pos_override is None else np.asarray(pos_override, np.int32)
    lens_d = torch.from_numpy(lens).cuda()
    pos_d = torch.from_numpy(pos).cuda()
    out = torch.full((c["B"], HQ, D), 7.0, dtype=torch.bfloat16, device="cuda")
    if append:
        eng.append(0, dev_bf16(c["k_new"]), dev_bf16(c["v_new"]), q, pos_d)
    eng.attention(0, q, lens_d, out)
    status, flag = eng.check_errors()
    res = dict(pool=u16(eng.slab.view(torch.bfloat16)), q=u16(q), out=u16(out), status=status, flag=flag)
    eng.close()
    return res


def oracle_run(c):
    pool = c["pool"].copy()
    q = c["q"].copy()
    g = oracle.geom(c["num_pages"])
    oracle.append(pool, g, c["bt"], c["seq_lens"] - 1, c["k_new"], c["v_new"], q)
    out_bf16, out_f64 = oracle.decode(pool, g, c["bt"], c["seq_lens"], q, SCALE)
    return dict(pool=pool, q=q, out=out_bf16, out_f64=out_f64)


def assert_close(gpu_u16, ref_f64):
    got = ph.bf16_to_f64(gpu_u16)
    err = np.abs(got - ref_f64)
    bound = ATOL + RTOL * np.abs(ref_f64)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"max excess at {worst}: got {got[worst]} ref {ref_f64[worst]}"


# ---------------------------------------------------------------------------- append

def test_rope_table_holds_cos_and_sin_to_48_bits():
    # entry (p, i) = {cos_hi, sin_hi, cos_lo, sin_lo}: hi the nearest FP32, hi + lo the
    # FP64 factor to about 2^-48 (the oracle's definition of the angle, R5/R6)
    max_pos = 2048
    t = pkv.rope_table(max_pos, "cuda", wl.ROPE_THETA).cpu().numpy().reshape(max_pos, D // 2, 4).astype(np.float64)
    p = np.arange(max_pos)[:, None]
    ang = p * np.array([oracle.rope_inv_freq(wl.ROPE_THETA, D, int(k)) for k in range(D // 2)])[None, :]
    c, s_ = np.cos(ang), np.sin(ang)
    assert np.array_equal(t[..., 0], c.astype(np.float32)) and np.array_equal(t[..., 1], s_.astype(np.float32))
    assert np.abs(t[..., 0] + t[..., 2] - c).max() <= 2.0**-47
    assert np.abs(t[..., 1] + t[..., 3] - s_).max() <= 2.0**-47


@pytest.mark.parametrize("seq_lens", [[17, 40], [1, 16, 17, 32, 33, 2048]])
def test_append_placement_bit_exact(seq_lens):
    c = make_case(1, seq_lens)
    g, o = gpu_run(c), oracle_run(c)
    changed_gpu = np.flatnonzero(g["pool"] != c["pool"])
    changed_ref = np.flatnonzero(o["pool"] != c["pool"])
    assert np.array_equal(changed_gpu, changed_ref)
    P_g, P_o = ph.pool_view(g["pool"]), ph.pool_view(o["pool"])
    for b, L in enumerate(c["seq_lens"]):
        page, slot = c["bt"][b, (L - 1) // PS], (L - 1) % PS
        assert np.array_equal(P_g[page, 1, :, slot], c["v_new"][b])            # V bit-exact
        assert ulp_distance(P_g[page, 0, :, slot], P_o[page, 0, :, slot]).max() <= 1
    assert ulp_distance(g["q"], o["q"]).max() <= 1


# ---------------------------------------------------------------------------- attention

@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_config(variant):
    c = make_case(12, [17, 40], num_pages=8)
    g, o = gpu_run(c, variant=variant), oracle_run(c)
    assert g["status"] == pkv.PKV_OK and g["flag"] == 0
    assert_close(g["out"], o["out_f64"])


RAGGED = [1, 2, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 1000, 2047, 2048]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("chunk", [1, 3, 16, 128])
def test_ragged_batch(variant, chunk):
    c = make_case(3, RAGGED, max_blocks=128)
    g, o = gpu_run(c, chunk=chunk, variant=variant), oracle_run(c)
    assert g["status"] == pkv.PKV_OK and g["flag"] == 0
    assert_close(g["out"], o["out_f64"])


@pytest.mark.parametrize("variant", VARIANTS)
def test_key_outliers(variant):
    # 1 % of cached key rows scaled by 8 stress the running-max tracking
    c = make_case(4, [300, 700, 64, 2048], max_blocks=128)
    rng = np.random.default_rng(44)
    P = ph.pool_view(c["pool"])
    mask = rng.random(P.shape[:1] + P.shape[2:4]) < 0.01
    keys = P[:, 0]
    keys[mask] = wl.scale_bf16_by_8(keys[mask])
    g, o = gpu_run(c, variant=variant), oracle_run(c)
    assert_close(g["out"], o["out_f64"])


@pytest.mark.parametrize("variant", VARIANTS)
def test_single_token_returns_v_exactly(variant):
    c = make_case(5, [1, 1, 1, 1])
    g = gpu_run(c, variant=variant)
    for b in range(4):
        for h in range(HQ):
            assert np.array_equal(g["out"][b, h], c["v_new"][b, h // 4])


@pytest.mark.parametrize("variant", VARIANTS)
def test_physical_page_order_is_irrelevant(variant):
    lens = [40, 300, 17, 129]
    a = gpu_run(make_case(6, lens, num_pages=64, perm_seed=100), variant=variant)
    b = gpu_run(make_case(6, lens, num_pages=64, perm_seed=200), variant=variant)
    assert np.array_equal(a["out"], b["out"])


@pytest.mark.parametrize("variant", VARIANTS)
def test_batch_invariance(variant):
    lens = [5, 700, 33, 2048, 16, 250]
    full = make_case(7, lens, max_blocks=128)
    g_full = gpu_run(full, chunk=8, variant=variant)
    for b in [0, 1, 3, 5]:
        one = {k: (v[b:b + 1] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == len(lens) else v)
               for k, v in full.items()}
        one["B"] = 1
        g_one = gpu_run(one, chunk=8, variant=variant)
        assert np.array_equal(g_one["out"][0], g_full["out"][b])


@pytest.mark.parametrize("variant", VARIANTS)
def test_chunking_agrees_to_rounding(variant):
    """One chunk per sequence vs one page per chunk.  The SIMT policy computes in
    FP32 throughout, so the two differ by FP32 rounding only (<= 2 BF16 ulps after
    the final rounding).  The MMA policy rounds each softmax weight p to BF16 (relative
    error <= 2^-9) relative to a running max that depends on the chunking, so the two
    outputs may differ by up to 2 * 2^-9 * max_t |v_t| plus the final rounding."""
    c = make_case(8, [2048, 1500, 129], max_blocks=128)
    one_chunk = gpu_run(c, chunk=128, variant=variant)
    per_page = gpu_run(c, chunk=1, variant=variant)
    if variant == pkv.PKV_DECODE_SIMT:
        assert ulp_distance(one_chunk["out"], per_page["out"]).max() <= 2
    else:
        a, b = ph.bf16_to_f64(one_chunk["out"]), ph.bf16_to_f64(per_page["out"])
        vmax = np.abs(ph.bf16_to_f64(c["V"])).max(axis=(2, 3))            # [B][Hkv]
        bound = 2 * 2.0**-9 * np.repeat(vmax, HQ // HKV, axis=1)[..., None] + 2.0**-7 * np.abs(a)
        assert np.all(np.abs(a - b) <= bound)


def test_variants_agree():
    c = make_case(9, RAGGED, max_blocks=128)
    a = ph.bf16_to_f64(gpu_run(c, variant=pkv.PKV_DECODE_SIMT)["out"])
    b = ph.bf16_to_f64(gpu_run(c, variant=pkv.PKV_DECODE_MMA)["out"])
    assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(a))


# ---------------------------------------------------------------------------- device bounds checks

@pytest.mark.parametrize("variant", VARIANTS)
def test_bad_page_id_sets_flag(variant):
    c = make_case(10, [40, 60])
    bad = c["bt"].copy()
    bad[1, 1] = c["num_pages"]          # outside the pool: checked before any copy
    c_bad = dict(c, bt=bad)
    g = gpu_run(c_bad, variant=variant, append=False, seq_lens_override=c["seq_lens"] - 1)
    assert g["status"] == pkv.PKV_ERR_DEVICE_BOUNDS and g["flag"] & pkv.PKV_DEVERR_PAGE_RANGE
    # the healthy sequence is still right
    o = oracle.decode(c["pool"], oracle.geom(c["num_pages"]), c["bt"], c["seq_lens"] - 1, c["q"], SCALE)[1]
    assert_close(g["out"][0], o[0])


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_length_sets_flag_and_zeros(variant):
    c = make_case(11, [20, 30])
    g = gpu_run(c, variant=variant, append=False, seq_lens_override=[0, 29])
    assert g["status"] == pkv.PKV_ERR_DEVICE_BOUNDS and g["flag"] & pkv.PKV_DEVERR_LENGTH
    assert np.all(g["out"][0] == 0)


def test_append_position_out_of_range_sets_flag():
    c = make_case(12, [20, 30])
    g = gpu_run(c, seq_lens_override=[19, 29], pos_override=[19, c["max_blocks"] * PS])
    assert g["flag"] & pkv.PKV_DEVERR_LENGTH
    # sequence 1 wrote nothing: only sequence 0's slots changed
    changed = np.flatnonzero(g["pool"] != c["pool"])
    assert changed.size == 2 * HKV * D


# ---------------------------------------------------------------------------- full-size, bench launch configuration

@pytest.mark.parametrize("name,layers", [("tiny", (0,)), ("b8", tuple(range(16))), ("b64", tuple(range(16))),
                                         ("b256", (0, 15))])
def test_full_size_every_unit(name, layers):
    # every (layer, sequence, query head) of a whole b8 / b64 step and of two whole b256
    # layers, at the benchmark's launch settings, against the oracle
    from tests import full_size

    checked = full_size.check_full_size(name, "bf16", layers)
    assert checked == wl.make_workload(name).batch * len(layers) * HQ
