"""CPU-only checks of libpkv: the library loads, exports every symbol the public
header declares, and its host-side logic (page pool allocator, block-table
builder, argument validation) behaves as documented.  No CUDA work is issued:
the pool functions are host only, and the launch entry points are only called
with arguments that fail validation before any CUDA call.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_decode_12_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
FAKE_SLAB = 0x7F0000000000  # never dereferenced by host code


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_12_gb300 import _build

    _build.build()


def header_functions(path=HEADER):
    text = open(path).read()
    return sorted(set(re.findall(r"^(?:int|size_t|const char \*)\s*(pkv_\w+)\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported():
    declared = header_functions()
    assert len(declared) >= 12
    lib = ctypes.CDLL(pkv.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(pkv.EXPORTED) == declared
    # the measurement header's probes are in the same library and bound by the binding
    probes = header_functions(os.path.join(ROOT, "include", "pkv_probe.h"))
    assert probes == sorted(pkv.EXPORTED_PROBE)
    for name in probes:
        assert hasattr(lib, name), name


def test_probe_validation_before_any_cuda_call():
    for fn in (pkv.pkv_probe_read_ldg, pkv.pkv_probe_read_bulk):
        for nbytes, sink, ctas in ((0, FAKE_SLAB, 1), (32768, None, 1), (32768 + 8, FAKE_SLAB, 1),
                                   (32768, FAKE_SLAB, 0), (32768, FAKE_SLAB, 9)):
            with pytest.raises(pkv.PkvError) as e:
                fn(FAKE_SLAB, nbytes, sink, ctas, 0)
            assert e.value.status == pkv.PKV_ERR_INVALID_ARG


def test_version_and_status_strings():
    assert "sm_103a" in pkv.pkv_version()
    assert pkv.status_string(pkv.PKV_OK) == "ok"
    assert "out of pages" in pkv.status_string(pkv.PKV_ERR_OUT_OF_PAGES)
    assert pkv.status_string(12345) == "unknown status"


def make_pool(pages, seed=1):
    return pkv.pkv_pool_create(FAKE_SLAB, pages * pkv.PKV_PAGE_BYTES, seed=seed)


def test_pool_create_validation():
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(FAKE_SLAB + 8, 4 * pkv.PKV_PAGE_BYTES)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(FAKE_SLAB, pkv.PKV_PAGE_BYTES - 1)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(FAKE_SLAB, 4 * pkv.PKV_PAGE_BYTES, page_size=32)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    with pytest.raises(pkv.PkvError):
        pkv.pkv_pool_create(None, 4 * pkv.PKV_PAGE_BYTES)


def test_pool_info_geometry():
    p = make_pool(10)
    info = pkv.pkv_pool_info(p)
    assert info["num_pages"] == 10 and info["num_free"] == 10
    assert info["k_base"] == FAKE_SLAB and info["v_base"] == FAKE_SLAB + 16384
    assert info["page_stride_bytes"] == 32768
    pkv.pkv_pool_destroy(p)


def test_alloc_all_or_nothing_and_free():
    p = make_pool(10)
    a = pkv.pkv_pool_alloc(p, 7)
    assert len(set(a.tolist())) == 7 and a.min() >= 0 and a.max() < 10
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_alloc(p, 4)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES
    assert pkv.pkv_pool_info(p)["num_free"] == 3          # nothing taken on failure
    pkv.pkv_pool_free(p, a[:2])
    assert pkv.pkv_pool_info(p)["num_free"] == 5
    rest = pkv.pkv_pool_alloc(p, 5)
    assert set(rest.tolist()) | set(a[2:].tolist()) == set(range(10))
    pkv.pkv_pool_destroy(p)


def test_free_errors_leave_pool_unchanged():
    p = make_pool(6)
    a = pkv.pkv_pool_alloc(p, 4)
    pkv.pkv_pool_free(p, a[:1])
    with pytest.raises(pkv.PkvError) as e:                 # a[0] already free
        pkv.pkv_pool_free(p, [a[1], a[0]])
    assert e.value.status == pkv.PKV_ERR_DOUBLE_FREE
    with pytest.raises(pkv.PkvError) as e:                 # repeated in one call
        pkv.pkv_pool_free(p, [a[2], a[2]])
    assert e.value.status == pkv.PKV_ERR_DOUBLE_FREE
    with pytest.raises(pkv.PkvError) as e:                 # foreign id
        pkv.pkv_pool_free(p, [a[3], 6])
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    assert pkv.pkv_pool_info(p)["num_free"] == 3
    pkv.pkv_pool_free(p, a[1:])                            # the failed calls freed nothing
    assert pkv.pkv_pool_info(p)["num_free"] == 6
    pkv.pkv_pool_destroy(p)


def test_block_tables_properties():
    p = make_pool(400, seed=5)
    lens = np.array([1, 16, 17, 32, 33, 0, 200], dtype=np.int32)
    bt = pkv.pkv_block_tables_build(p, 3, lens, 16)
    need = -(-lens // 16)
    used = []
    for layer in range(3):
        for b, n in enumerate(need):
            row = bt[layer, b]
            assert np.all(row[:n] >= 0) and np.all(row[:n] < 400)
            assert np.all(row[n:] == -1)
            used.extend(row[:n].tolist())
    assert len(used) == len(set(used)) == 3 * need.sum()     # no page shared between rows
    assert pkv.pkv_pool_info(p)["num_free"] == 400 - 3 * need.sum()
    # pages are scattered through the slab, not handed out in order
    assert sorted(used) != used
    pkv.pkv_pool_destroy(p)


def test_block_tables_seeded_and_all_or_nothing():
    lens = np.array([100, 50], dtype=np.int32)
    a = pkv.pkv_block_tables_build(make_pool(64, seed=9), 2, lens, 8)
    b = pkv.pkv_block_tables_build(make_pool(64, seed=9), 2, lens, 8)
    c = pkv.pkv_block_tables_build(make_pool(64, seed=10), 2, lens, 8)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    p = make_pool(20)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_block_tables_build(p, 2, lens, 8)          # needs 22 pages
    assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES
    assert pkv.pkv_pool_info(p)["num_free"] == 20
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_block_tables_build(p, 1, np.array([129], np.int32), 8)   # 9 pages > 8
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_block_tables_build(p, 1, np.array([-1], np.int32), 8)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG


def test_workspace_bytes():
    # B x 8 merge counters, then B x 32 heads x chunks x (m, l) floats, each 256-aligned,
    # then x 64 floats of o; the fused step uses the same layout
    def align(x):
        return (x + 255) // 256 * 256

    for B, max_blocks, ppc in ((256, 128, 16), (3, 100, 7), (1, 1, 1)):
        chunks = -(-max_blocks // ppc)
        want = align(B * 8 * 4) + align(B * 32 * chunks * 8) + B * 32 * chunks * 64 * 4
        assert pkv.pkv_decode_workspace_bytes(B, max_blocks, ppc) == want
        assert pkv.pkv_decode_step_workspace_bytes(B, max_blocks, ppc) == want
    assert pkv.pkv_decode_workspace_bytes(0, 128, 16) == 0


def test_rope_table_bytes():
    # 16 bytes per (position, pair): cos and sin, each as a high and a low FP32 part
    assert pkv.pkv_rope_table_bytes(2048, 32) == 2048 * 32 * 16
    assert pkv.pkv_rope_table_bytes(1, 32) == 512
    assert pkv.pkv_rope_table_bytes(0, 32) == 0 and pkv.pkv_rope_table_bytes(2048, 16) == 0


def test_launch_entry_points_validate_before_any_cuda_call():
    p = make_pool(8)
    dummy = FAKE_SLAB
    with pytest.raises(pkv.PkvError) as e:     # B = 0
        pkv.pkv_decode_attention(p, dummy, dummy, 128, dummy, 0, 0.125, 16, dummy, 1 << 20, dummy, None, 0)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:     # chunk of 0 pages
        pkv.pkv_decode_attention(p, dummy, dummy, 128, dummy, 4, 0.125, 0, dummy, 1 << 20, dummy, None, 0)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:     # workspace too small
        pkv.pkv_decode_attention(p, dummy, dummy, 128, dummy, 4, 0.125, 16, dummy, 64, dummy, None, 0)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE_TOO_SMALL
    for variant in (9, 0x400, 0x800, 0x10000, pkv.PKV_DECODE_SPLIT_MERGE | pkv.PKV_STEP_SORTED,
                    pkv.PKV_DECODE_SPLIT_MERGE | pkv.PKV_STEP_TEST_EXPIRE_WAIT, pkv.PKV_STEP_RING(1),
                    pkv.PKV_STEP_RING(5)):
        with pytest.raises(pkv.PkvError) as e:     # unknown variant or option
            pkv.pkv_decode_attention_variant(p, dummy, dummy, 128, dummy, 4, 0.125, 16, dummy, 1 << 20, dummy,
                                             None, 0, variant=variant)
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG, hex(variant)
    with pytest.raises(pkv.PkvError) as e:     # misaligned k_new
        pkv.pkv_append_rope(p, dummy + 2, dummy, None, dummy, 128, dummy, 4, dummy, 2048, None, 0)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:     # half_dim other than 32
        pkv.pkv_rope_table_init(500000.0, 2048, 16, dummy, 0)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    pkv.pkv_pool_destroy(p)


def test_fp8_pool_geometry_and_format():
    assert pkv.PKV_PAGE_BYTES_FP8 == 17408
    p = pkv.pkv_pool_create_fp8(FAKE_SLAB, 10 * pkv.PKV_PAGE_BYTES_FP8 + 100, seed=3)
    info = pkv.pkv_pool_info(p)
    assert info["num_pages"] == 10 and info["num_free"] == 10
    assert info["k_base"] == FAKE_SLAB and info["v_base"] == FAKE_SLAB + 1024   # head 0: K rows, then V rows
    assert info["page_stride_bytes"] == 17408
    assert pkv.pkv_pool_kv_format(p) == pkv.PKV_KV_FP8
    b = make_pool(2)
    assert pkv.pkv_pool_kv_format(b) == pkv.PKV_KV_BF16
    # same allocator: the seeded shuffle hands out the same ids as a BF16 pool
    q = make_pool(10, seed=3)
    assert np.array_equal(pkv.pkv_pool_alloc(p, 10), pkv.pkv_pool_alloc(q, 10))
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create_fp8(FAKE_SLAB + 8, 4 * pkv.PKV_PAGE_BYTES_FP8)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create_fp8(FAKE_SLAB, pkv.PKV_PAGE_BYTES_FP8 - 1)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    for x in (p, b, q):
        pkv.pkv_pool_destroy(x)


def test_fp8_pool_rejects_unsupported_options_before_any_cuda_call():
    p = pkv.pkv_pool_create_fp8(FAKE_SLAB, 8 * pkv.PKV_PAGE_BYTES_FP8)
    dummy = FAKE_SLAB
    with pytest.raises(pkv.PkvError) as e:     # SIMT policy has no FP8 form
        pkv.pkv_decode_attention_variant(p, dummy, dummy, 128, dummy, 4, 0.125, 16, dummy, 1 << 20, dummy, None,
                                         0, variant=pkv.PKV_DECODE_SIMT)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    ws = pkv.pkv_decode_step_workspace_bytes(4, 128, 16)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step(p, dummy, dummy, dummy, dummy, 128, dummy, 4, dummy, 2048, 0.125, 16, dummy, ws,
                            dummy, None, 0, options=pkv.PKV_DECODE_SIMT)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    pkv.pkv_pool_destroy(p)


def test_step_options_validation_before_any_cuda_call():
    p = make_pool(8)
    dummy = FAKE_SLAB
    ws = pkv.pkv_decode_step_workspace_bytes(1025, 128, 16)
    # more sequences than the sorted order handles; bits of schedules that no longer
    # exist (0x400, 0x800) or of the removed early trigger (0x10000); the two-kernel
    # attention form is not a step option; ring depths outside 2..4
    for B, opt in ((1025, pkv.PKV_STEP_SORTED), (4, 0x400), (4, 0x800), (4, 0x10000),
                   (4, pkv.PKV_DECODE_SPLIT_MERGE), (4, pkv.PKV_STEP_RING(1)), (4, pkv.PKV_STEP_RING(7))):
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_decode_step(p, dummy, dummy, dummy, dummy, 128, dummy, B, dummy, 2048, 0.125, 16, dummy, ws,
                                dummy, None, 0, options=opt)
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG, (B, hex(opt))
    pkv.pkv_pool_destroy(p)


def test_step_layers_validation_before_any_cuda_call():
    p = make_pool(8)
    dummy = FAKE_SLAB
    ws = pkv.pkv_decode_step_workspace_bytes(4, 128, 16)
    args = (dummy, dummy, dummy, dummy, 128, dummy, 4, dummy, 2048, 0.125, 16, dummy, ws, dummy, None, 0)
    bad = [dict(layers=0), dict(layers=2, kv_layer_stride=-512), dict(layers=2, q_layer_stride=-1),
           dict(layers=2, bt_layer_stride=-128), dict(layers=2, kv_layer_stride=3),   # 6-byte layer step
           dict(layers=2, q_layer_stride=4100)]
    for kw in bad:
        layers = kw.pop("layers")
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_decode_step_layers(p, layers, *args, **kw)
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG, kw
    # layer 0 is validated as pkv_decode_step validates it: a bad batch launches nothing
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step_layers(p, 16, dummy, dummy, dummy, dummy, 128, dummy, 0, dummy, 2048, 0.125, 16, dummy,
                                   ws, dummy, None, 0, kv_layer_stride=4 * 512, q_layer_stride=4 * 2048,
                                   bt_layer_stride=4 * 128)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    pkv.pkv_pool_destroy(p)
