"""Thin ctypes binding of ``libpkv.so`` (C ABI declared in ``include/pkv.h``).

Functions keep the C names and argument order.  Marshalling only: torch tensors
are passed as raw device pointers (``data_ptr``), streams as the raw
``cudaStream_t`` of ``torch.cuda.current_stream()`` unless one is given, and
every status code is turned into a ``PkvError``.  All computation happens in
the library's CUDA kernels; there is no fallback.  If ``libpkv.so`` has not
been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
# PKV_LIBRARY selects another build of the same ABI (e.g. libpkv_timeline.so)
LIB_PATH = os.environ.get("PKV_LIBRARY") or os.path.join(HERE, "libpkv.so")

PKV_PAGE_SIZE = 16
PKV_NUM_Q_HEADS = 32
PKV_NUM_KV_HEADS = 8
PKV_HEAD_DIM = 64
PKV_PAGE_BYTES = 2 * PKV_NUM_KV_HEADS * PKV_PAGE_SIZE * PKV_HEAD_DIM * 2

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_OUT_OF_PAGES = -2
PKV_ERR_DOUBLE_FREE = -3
PKV_ERR_CUDA = -4
PKV_ERR_DEVICE_BOUNDS = -5
PKV_ERR_BUDGET_EXCEEDS_POOL = -6
PKV_ERR_UNSUPPORTED = -7
PKV_ERR_WORKSPACE_TOO_SMALL = -8

PKV_DEVERR_PAGE_RANGE = 0x1
PKV_DEVERR_LENGTH = 0x2
PKV_DEVERR_TIMEOUT = 0x4

PKV_DECODE_DEFAULT = 0
PKV_DECODE_SIMT = 1
PKV_DECODE_MMA = 2
PKV_STEP_NO_PDL = 0x100
PKV_STEP_GRID = 0x200
PKV_STEP_RING_MASK = 0xF000
PKV_STEP_SORTED = 0x20000
PKV_STEP_TEST_EXPIRE_WAIT = 0x40000
PKV_DECODE_SPLIT_MERGE = 0x80000


def PKV_STEP_RING(n: int) -> int:
    return n << 12

# every symbol include/pkv.h declares
EXPORTED = (
    "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_alloc", "pkv_pool_free", "pkv_pool_info",
    "pkv_block_tables_build", "pkv_rope_table_bytes", "pkv_rope_table_init", "pkv_append_rope",
    "pkv_decode_workspace_bytes",
    "pkv_decode_attention", "pkv_decode_attention_variant", "pkv_decode_attention_noalloc",
    "pkv_decode_step_workspace_bytes", "pkv_decode_step", "pkv_decode_step_layers", "pkv_check_device_error",
    "pkv_status_string", "pkv_version",
)


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i32p = ctypes.POINTER(ctypes.c_int32)


def lib():
    """Load libpkv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                           f"g.build()'` (or python -m paged_kv_decode_12_gb300._build)")
    L = ctypes.CDLL(LIB_PATH)
    L.pkv_pool_create.argtypes = [_vp, ctypes.c_size_t, _i32, _i32, _i32, ctypes.c_uint64, ctypes.POINTER(_vp)]
    L.pkv_pool_destroy.argtypes = [_vp]
    L.pkv_pool_alloc.argtypes = [_vp, _i32, _i32p]
    L.pkv_pool_free.argtypes = [_vp, _i32, _i32p]
    L.pkv_pool_info.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_int64),
                                ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
    L.pkv_block_tables_build.argtypes = [_vp, _i32, _i32, _i32p, _i32, _i32p]
    L.pkv_rope_table_bytes.argtypes = [_i32, _i32]
    L.pkv_rope_table_bytes.restype = ctypes.c_size_t
    L.pkv_rope_table_init.argtypes = [ctypes.c_double, _i32, _i32, _vp, _vp]
    L.pkv_append_rope.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp]
    L.pkv_decode_workspace_bytes.argtypes = [_i32, _i32, _i32]
    L.pkv_decode_workspace_bytes.restype = ctypes.c_size_t
    L.pkv_decode_attention.argtypes = [_vp, _vp, _vp, _i32, _vp, _i32, ctypes.c_float, _i32, _vp,
                                       ctypes.c_size_t, _vp, _vp, _vp]
    L.pkv_decode_attention_variant.argtypes = L.pkv_decode_attention.argtypes + [_i32]
    L.pkv_decode_attention_noalloc.argtypes = [_vp, _vp, _vp, _i32, _vp, _i32, ctypes.c_float, _i32, _vp, _vp,
                                               _vp]
    L.pkv_decode_step_workspace_bytes.argtypes = [_i32, _i32, _i32]
    L.pkv_decode_step_workspace_bytes.restype = ctypes.c_size_t
    L.pkv_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _i32, ctypes.c_float, _i32, _vp,
                                  ctypes.c_size_t, _vp, _vp, _vp, _i32]
    L.pkv_decode_step_layers.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _i32, ctypes.c_float,
                                         _i32, _vp, ctypes.c_size_t, _vp, _vp, _vp, _i32, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64]
    L.pkv_check_device_error.argtypes = [_vp, _i32p, _vp]
    L.pkv_status_string.argtypes = [_i32]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_version.argtypes = []
    L.pkv_version.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name not in ("pkv_decode_workspace_bytes", "pkv_decode_step_workspace_bytes", "pkv_rope_table_bytes",
                        "pkv_status_string", "pkv_version"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


# ---------------------------------------------------------------------------- marshalling

def _ptr(x):
    """Device/host pointer from a tensor, an int address or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str) -> int:
    if status != PKV_OK:
        raise PkvError(status, what)
    return status


def _np_i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def status_string(status: int) -> str:
    try:
        return lib().pkv_status_string(int(status)).decode()
    except RuntimeError:
        return "unknown"


pkv_status_string = status_string


def pkv_version() -> str:
    return lib().pkv_version().decode()


# ---------------------------------------------------------------------------- pool

def pkv_pool_create(dev_slab, slab_bytes: int, page_size: int = PKV_PAGE_SIZE,
                    num_kv_heads: int = PKV_NUM_KV_HEADS, head_dim: int = PKV_HEAD_DIM, seed: int = 0):
    """Returns an opaque pool handle (ctypes.c_void_p)."""
    out = ctypes.c_void_p()
    _check(lib().pkv_pool_create(_ptr(dev_slab), int(slab_bytes), page_size, num_kv_heads, head_dim,
                                 int(seed) & (2**64 - 1), ctypes.byref(out)), "pkv_pool_create")
    return out


def pkv_pool_destroy(pool) -> None:
    _check(lib().pkv_pool_destroy(pool), "pkv_pool_destroy")


def pkv_pool_alloc(pool, n: int) -> np.ndarray:
    ids = np.empty(max(n, 0), dtype=np.int32)
    _check(lib().pkv_pool_alloc(pool, int(n), ids.ctypes.data_as(_i32p)), "pkv_pool_alloc")
    return ids


def pkv_pool_free(pool, ids) -> None:
    ids = _np_i32(ids)
    _check(lib().pkv_pool_free(pool, ids.size, ids.ctypes.data_as(_i32p)), "pkv_pool_free")


def pkv_pool_info(pool) -> dict:
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    stride = ctypes.c_int64()
    n, free = ctypes.c_int(), ctypes.c_int()
    _check(lib().pkv_pool_info(pool, ctypes.byref(k), ctypes.byref(v), ctypes.byref(stride), ctypes.byref(n),
                               ctypes.byref(free)), "pkv_pool_info")
    return {"k_base": k.value, "v_base": v.value, "page_stride_bytes": stride.value, "num_pages": n.value,
            "num_free": free.value}


def pkv_block_tables_build(pool, layers: int, seq_lens, max_blocks: int) -> np.ndarray:
    """Host block tables int32 [layers][B][max_blocks]."""
    seq_lens = _np_i32(seq_lens)
    B = seq_lens.size
    bt = np.empty((layers, B, max_blocks), dtype=np.int32)
    _check(lib().pkv_block_tables_build(pool, layers, B, seq_lens.ctypes.data_as(_i32p), max_blocks,
                                        bt.ctypes.data_as(_i32p)), "pkv_block_tables_build")
    return bt


# ---------------------------------------------------------------------------- RoPE / append / decode

def pkv_rope_table_bytes(max_pos: int, half_dim: int) -> int:
    return int(lib().pkv_rope_table_bytes(max_pos, half_dim))


def rope_table(max_pos: int, device, theta: float = 500000.0, half_dim: int = PKV_HEAD_DIM // 2):
    """A device float32 tensor of pkv_rope_table_bytes(...) bytes, filled by pkv_rope_table_init."""
    import torch

    t = torch.empty(pkv_rope_table_bytes(max_pos, half_dim) // 4, dtype=torch.float32, device=device)
    pkv_rope_table_init(theta, max_pos, half_dim, t)
    return t


def pkv_rope_table_init(theta: float, max_pos: int, half_dim: int, dev_cos_sin, stream=None) -> None:
    _check(lib().pkv_rope_table_init(float(theta), max_pos, half_dim, _ptr(dev_cos_sin), _stream(stream)),
           "pkv_rope_table_init")


def pkv_append_rope(pool, k_new, v_new, q, bt_dev, max_blocks: int, pos_dev, B: int, rope_table, max_pos: int,
                    dev_err_flag=None, stream=None) -> None:
    _check(lib().pkv_append_rope(pool, _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(bt_dev), max_blocks,
                                 _ptr(pos_dev), B, _ptr(rope_table), max_pos, _ptr(dev_err_flag),
                                 _stream(stream)), "pkv_append_rope")


def pkv_decode_workspace_bytes(B: int, max_blocks: int, pages_per_chunk: int) -> int:
    return int(lib().pkv_decode_workspace_bytes(B, max_blocks, pages_per_chunk))


def pkv_decode_attention(pool, q, bt_dev, max_blocks: int, seq_lens_dev, B: int, scale: float,
                         pages_per_chunk: int, workspace, workspace_bytes: int, out, dev_err_flag=None,
                         stream=None) -> None:
    _check(lib().pkv_decode_attention(pool, _ptr(q), _ptr(bt_dev), max_blocks, _ptr(seq_lens_dev), B,
                                      float(scale), pages_per_chunk, _ptr(workspace), int(workspace_bytes),
                                      _ptr(out), _ptr(dev_err_flag), _stream(stream)), "pkv_decode_attention")


def pkv_decode_attention_variant(pool, q, bt_dev, max_blocks: int, seq_lens_dev, B: int, scale: float,
                                 pages_per_chunk: int, workspace, workspace_bytes: int, out, dev_err_flag=None,
                                 stream=None, variant: int = PKV_DECODE_DEFAULT) -> None:
    _check(lib().pkv_decode_attention_variant(pool, _ptr(q), _ptr(bt_dev), max_blocks, _ptr(seq_lens_dev), B,
                                              float(scale), pages_per_chunk, _ptr(workspace),
                                              int(workspace_bytes), _ptr(out), _ptr(dev_err_flag),
                                              _stream(stream), int(variant)),
           "pkv_decode_attention_variant")


def pkv_decode_step_workspace_bytes(B: int, max_blocks: int, pages_per_chunk: int) -> int:
    return int(lib().pkv_decode_step_workspace_bytes(B, max_blocks, pages_per_chunk))


def pkv_decode_step(pool, k_new, v_new, q, bt_dev, max_blocks: int, seq_lens_dev, B: int, rope_table,
                    max_pos: int, scale: float, pages_per_chunk: int, workspace, workspace_bytes: int, out,
                    dev_err_flag=None, stream=None, options: int = PKV_DECODE_DEFAULT) -> None:
    _check(lib().pkv_decode_step(pool, _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(bt_dev), max_blocks,
                                 _ptr(seq_lens_dev), B, _ptr(rope_table), max_pos, float(scale), pages_per_chunk,
                                 _ptr(workspace), int(workspace_bytes), _ptr(out), _ptr(dev_err_flag),
                                 _stream(stream), int(options)), "pkv_decode_step")


def pkv_decode_step_layers(pool, layers: int, k_new, v_new, q, bt_dev, max_blocks: int, seq_lens_dev, B: int,
                           rope_table, max_pos: int, scale: float, pages_per_chunk: int, workspace,
                           workspace_bytes: int, out, dev_err_flag=None, stream=None,
                           options: int = PKV_DECODE_DEFAULT, kv_layer_stride: int = 0, q_layer_stride: int = 0,
                           bt_layer_stride: int = 0) -> None:
    """pkv_decode_step for every layer in one call; strides in elements (see include/pkv.h)."""
    _check(lib().pkv_decode_step_layers(pool, int(layers), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(bt_dev),
                                        max_blocks, _ptr(seq_lens_dev), B, _ptr(rope_table), max_pos, float(scale),
                                        pages_per_chunk, _ptr(workspace), int(workspace_bytes), _ptr(out),
                                        _ptr(dev_err_flag), _stream(stream), int(options), int(kv_layer_stride),
                                        int(q_layer_stride), int(bt_layer_stride)), "pkv_decode_step_layers")


PKV_NOALLOC_SCRATCH_BYTES = 32 << 20


def pkv_decode_attention_noalloc(pool, q, bt_dev, max_blocks: int, seq_lens_dev, B: int, scale: float,
                                 pages_per_chunk: int, out, dev_err_flag=None, stream=None) -> None:
    """pkv_decode_attention with the library's static scratch instead of a workspace,
    for callers that cannot allocate device memory (see include/pkv.h)."""
    _check(lib().pkv_decode_attention_noalloc(pool, _ptr(q), _ptr(bt_dev), max_blocks, _ptr(seq_lens_dev), B,
                                              float(scale), pages_per_chunk, _ptr(out), _ptr(dev_err_flag),
                                              _stream(stream)), "pkv_decode_attention_noalloc")


def pkv_check_device_error(dev_err_flag, stream=None):
    """Synchronise the stream; returns (status, flag bits)."""
    flag = ctypes.c_int32(0)
    st = lib().pkv_check_device_error(_ptr(dev_err_flag), ctypes.byref(flag), _stream(stream))
    if st not in (PKV_OK, PKV_ERR_DEVICE_BOUNDS):
        raise PkvError(st, "pkv_check_device_error")
    return st, int(flag.value)


# ---------------------------------------------------------------------------- scheduler, prefill

PKV_SCHED_CONTINUOUS = 0
PKV_SCHED_STATIC = 1

EXPORTED = EXPORTED + (
    "pkv_sched_create", "pkv_sched_destroy", "pkv_sched_submit", "pkv_sched_admit", "pkv_sched_decode_batch",
    "pkv_sched_finish", "pkv_sched_get_stats", "pkv_prefill_append",
)


class SchedStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "pool_pages", "peak_active", "max_decode_batch", "peak_allocated_pages", "admission_waits",
        "final_free_pages", "submitted", "admitted", "finished", "rejected", "active", "waiting",
        "allocated_pages", "free_credits")]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


_lib_core = lib
_i64p = ctypes.POINTER(ctypes.c_int64)


def lib():  # noqa: F811 -- extends the loader with the scheduler and prefill signatures
    L = _lib_core()
    if not getattr(L, "_pkv_sched_bound", False):
        L.pkv_sched_create.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_vp)]
        L.pkv_sched_destroy.argtypes = [_vp]
        L.pkv_sched_submit.argtypes = [_vp, ctypes.c_int64, _i32, _i32]
        L.pkv_sched_admit.argtypes = [_vp, _i32, _i64p, _i32p, _i32p, ctypes.POINTER(_i32)]
        L.pkv_sched_decode_batch.argtypes = [_vp, _i32, _i64p, _i32p, _i32p, ctypes.POINTER(_i32)]
        L.pkv_sched_finish.argtypes = [_vp, ctypes.c_int64]
        L.pkv_sched_get_stats.argtypes = [_vp, ctypes.POINTER(SchedStats)]
        L.pkv_prefill_append.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]
        for name in ("pkv_sched_create", "pkv_sched_destroy", "pkv_sched_submit", "pkv_sched_admit",
                     "pkv_sched_decode_batch", "pkv_sched_finish", "pkv_sched_get_stats", "pkv_prefill_append"):
            getattr(L, name).restype = ctypes.c_int
        L._pkv_sched_bound = True
    return L


def pkv_sched_create(pool, layers: int, max_blocks: int, max_context: int, max_batch: int,
                     mode: int = PKV_SCHED_CONTINUOUS):
    out = ctypes.c_void_p()
    _check(lib().pkv_sched_create(pool, layers, max_blocks, max_context, max_batch, mode, ctypes.byref(out)),
           "pkv_sched_create")
    return out


def pkv_sched_destroy(sched) -> None:
    _check(lib().pkv_sched_destroy(sched), "pkv_sched_destroy")


def pkv_sched_submit(sched, rid: int, prompt_tokens: int, max_new_tokens: int) -> None:
    _check(lib().pkv_sched_submit(sched, int(rid), int(prompt_tokens), int(max_new_tokens)), "pkv_sched_submit")


def _out_array(given, size: int, dtype):
    """A caller's output array (C-contiguous, of ``dtype``, at least ``size`` elements), flat."""
    if given is None:
        return np.empty(size, dtype=dtype)
    flat = given.reshape(-1)
    if flat.dtype != dtype or flat.size < size or not flat.flags["C_CONTIGUOUS"] or not np.shares_memory(flat, given):
        raise ValueError(f"output array must be C-contiguous {np.dtype(dtype).name} with >= {size} elements")
    return flat


def pkv_sched_admit(sched, max_n: int, layers: int, max_blocks: int, ids_out=None, lens_out=None, bt_out=None):
    """Returns (ids int64 [n], prompt_lens int32 [n], bt_rows int32 [n][layers][max_blocks]),
    written into the given arrays (e.g. views of pinned host memory) if any."""
    ids = _out_array(ids_out, max_n, np.int64)
    lens = _out_array(lens_out, max_n, np.int32)
    bt = _out_array(bt_out, max_n * layers * max_blocks, np.int32).reshape(max_n, layers, max_blocks)
    n = ctypes.c_int(0)
    _check(lib().pkv_sched_admit(sched, max_n, ids.ctypes.data_as(_i64p), lens.ctypes.data_as(_i32p),
                                 bt.ctypes.data_as(_i32p), ctypes.byref(n)), "pkv_sched_admit")
    return ids[:n.value], lens[:n.value], bt[:n.value]


def pkv_sched_decode_batch(sched, max_b: int, layers: int, max_blocks: int, ids_out=None, lens_out=None,
                           bt_out=None):
    """Returns (ids int64 [B], seq_lens int32 [B], bt int32 [layers][B][max_blocks]), written
    into the given arrays (e.g. views of pinned host memory) if any; bt is compact: layer l's
    rows start at l * B * max_blocks."""
    ids = _out_array(ids_out, max_b, np.int64)
    lens = _out_array(lens_out, max_b, np.int32)
    bt = _out_array(bt_out, layers * max_b * max_blocks, np.int32)
    B = ctypes.c_int(0)
    _check(lib().pkv_sched_decode_batch(sched, max_b, ids.ctypes.data_as(_i64p), lens.ctypes.data_as(_i32p),
                                        bt.ctypes.data_as(_i32p), ctypes.byref(B)), "pkv_sched_decode_batch")
    b = B.value
    return ids[:b], lens[:b], bt[: layers * b * max_blocks].reshape(layers, b, max_blocks)


def pkv_sched_finish(sched, rid: int) -> None:
    _check(lib().pkv_sched_finish(sched, int(rid)), "pkv_sched_finish")


def pkv_sched_get_stats(sched) -> dict:
    st = SchedStats()
    _check(lib().pkv_sched_get_stats(sched, ctypes.byref(st)), "pkv_sched_get_stats")
    return st.as_dict()


def pkv_prefill_append(pool, k, v, bt_rows_dev, max_blocks: int, layers: int, start_pos: int, T: int, rope_table,
                       max_pos: int, dev_err_flag=None, stream=None) -> None:
    _check(lib().pkv_prefill_append(pool, _ptr(k), _ptr(v), _ptr(bt_rows_dev), max_blocks, layers, start_pos, T,
                                    _ptr(rope_table), max_pos, _ptr(dev_err_flag), _stream(stream)),
           "pkv_prefill_append")


# ---------------------------------------------------------------------------- FP8 pages

PKV_KV_BF16 = 0
PKV_KV_FP8 = 1
PKV_PAGE_BYTES_FP8 = 2 * PKV_NUM_KV_HEADS * PKV_PAGE_SIZE * (PKV_HEAD_DIM + 4)

EXPORTED = EXPORTED + ("pkv_pool_create_fp8", "pkv_pool_kv_format")

_lib_sched = lib


def lib():  # noqa: F811 -- extends the loader with the FP8 pool signatures
    L = _lib_sched()
    if not getattr(L, "_pkv_fp8_bound", False):
        L.pkv_pool_create_fp8.argtypes = [_vp, ctypes.c_size_t, ctypes.c_uint64, ctypes.POINTER(_vp)]
        L.pkv_pool_create_fp8.restype = ctypes.c_int
        L.pkv_pool_kv_format.argtypes = [_vp]
        L.pkv_pool_kv_format.restype = ctypes.c_int
        L._pkv_fp8_bound = True
    return L


def pkv_pool_create_fp8(dev_slab, slab_bytes: int, seed: int = 0):
    """Pool of FP8 E4M3 pages (codes + per-row FP32 scales); opaque handle."""
    out = ctypes.c_void_p()
    _check(lib().pkv_pool_create_fp8(_ptr(dev_slab), int(slab_bytes), int(seed) & (2**64 - 1), ctypes.byref(out)),
           "pkv_pool_create_fp8")
    return out


def pkv_pool_kv_format(pool) -> int:
    st = lib().pkv_pool_kv_format(pool)
    if st < 0:
        raise PkvError(st, "pkv_pool_kv_format")
    return st


# ---------------------------------------------------------------------------- read-bandwidth probes

# every symbol include/pkv_probe.h declares (a measurement aid, not the decode path)
EXPORTED_PROBE = ("pkv_probe_read_ldg", "pkv_probe_read_bulk")

_lib_fp8 = lib


def lib():  # noqa: F811 -- extends the loader with the probe signatures
    L = _lib_fp8()
    if not getattr(L, "_pkv_probe_bound", False):
        for name in EXPORTED_PROBE:
            getattr(L, name).argtypes = [_vp, ctypes.c_size_t, _vp, _i32, _vp]
            getattr(L, name).restype = ctypes.c_int
        L._pkv_probe_bound = True
    return L


def pkv_probe_read_ldg(buf, nbytes: int, sink, ctas_per_sm: int = 2, stream=None) -> None:
    _check(lib().pkv_probe_read_ldg(_ptr(buf), int(nbytes), _ptr(sink), int(ctas_per_sm), _stream(stream)),
           "pkv_probe_read_ldg")


def pkv_probe_read_bulk(buf, nbytes: int, sink, ctas_per_sm: int = 2, stream=None) -> None:
    _check(lib().pkv_probe_read_bulk(_ptr(buf), int(nbytes), _ptr(sink), int(ctas_per_sm), _stream(stream)),
           "pkv_probe_read_bulk")
