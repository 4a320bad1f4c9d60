"""FP64 CPU oracle for the paged-KV decode path (ctypes front end).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only callers allowed.  The
product library never imports this package and shares no code with it.

Every function marshals numpy arrays into the C oracle (``pkv_oracle.c``), which
restates the pages' definitions in plain FP64 loops; see that file's header for
the sources and the readings taken where the pages are silent.

Arrays of BF16 values are passed as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class OracleError(RuntimeError):
    pass


class PoolGeom(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
    ]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    gp = ctypes.POINTER(PoolGeom)
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_rope_inv_freq.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_rope_inv_freq.restype = ctypes.c_double
    lib.oracle_rope_rotate.argtypes = [f64p, ctypes.c_int, ctypes.c_longlong, ctypes.c_double, f64p]
    lib.oracle_rope_rotate.restype = None
    lib.oracle_pool_index.argtypes = [gp] + [ctypes.c_int] * 5
    lib.oracle_pool_index.restype = ctypes.c_int64
    lib.oracle_append.argtypes = [u16p, gp, i32p, ctypes.c_int, i32p, ctypes.c_int, u16p, u16p,
                                  u16p, ctypes.c_int, ctypes.c_double]
    lib.oracle_append.restype = ctypes.c_int
    lib.oracle_decode_one.argtypes = [u16p, gp, i32p, ctypes.c_int, ctypes.c_int, u16p, ctypes.c_int,
                                      ctypes.c_double, f64p, f64p]
    lib.oracle_decode_one.restype = ctypes.c_int
    lib.oracle_decode.argtypes = [u16p, gp, i32p, ctypes.c_int, i32p, ctypes.c_int, u16p, ctypes.c_int,
                                  ctypes.c_double, u16p, f64p]
    lib.oracle_decode.restype = ctypes.c_int
    lib.oracle_decode_contiguous.argtypes = [f64p, f64p, ctypes.c_int, i32p, ctypes.c_int, f64p,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                             f64p]
    lib.oracle_decode_contiguous.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(status: int, what: str):
    if status != 0:
        raise OracleError(f"{what} failed with status {status}")


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


# --------------------------------------------------------------------------- BF16

def bf16_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 values (exact)."""
    lib = _load()
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    flat_in, flat_out = b.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.oracle_bf16_to_double(int(flat_in[i]))
    return out


def bf16_from_f64(values) -> np.ndarray:
    """float64 values -> BF16 bit patterns, one round-to-nearest-even step."""
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_in, flat_out = v.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.oracle_bf16_from_double(float(flat_in[i]))
    return out


# --------------------------------------------------------------------------- RoPE

def rope_inv_freq(theta: float, head_dim: int, i: int) -> float:
    return _load().oracle_rope_inv_freq(float(theta), int(head_dim), int(i))


def rope_rotate(x, pos: int, theta: float) -> np.ndarray:
    """Rotate one head vector (float64, length head_dim) to absolute position pos."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib.oracle_rope_rotate(_ptr(x, ctypes.c_double), x.size, int(pos), float(theta),
                           _ptr(y, ctypes.c_double))
    return y


# --------------------------------------------------------------------------- pool

def geom(num_pages: int, page_size: int = 16, num_kv_heads: int = 8, head_dim: int = 64) -> PoolGeom:
    return PoolGeom(num_pages, page_size, num_kv_heads, head_dim)


def pool_index(g: PoolGeom, page: int, kv: int, head: int, slot: int, dim: int) -> int:
    return int(_load().oracle_pool_index(ctypes.byref(g), page, kv, head, slot, dim))


def append(pool: np.ndarray, g: PoolGeom, bt, pos, k_new, v_new, q=None, num_q_heads: int = 32,
           theta: float = 500000.0):
    """Append one token per sequence into ``pool`` (uint16, modified in place).

    bt: [B][max_blocks] int32; pos: [B]; k_new, v_new: [B][Hkv][D] uint16;
    q: [B][Hq][D] uint16 rotated in place when given.  Returns q.
    """
    lib = _load()
    assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
    bt = _i32(bt)
    pos = _i32(pos)
    k_new, v_new = _u16(k_new), _u16(v_new)
    B, max_blocks = bt.shape
    if q is not None:
        assert q.dtype == np.uint16 and q.flags["C_CONTIGUOUS"]
    st = lib.oracle_append(_ptr(pool, ctypes.c_uint16), ctypes.byref(g), _ptr(bt, ctypes.c_int32),
                           max_blocks, _ptr(pos, ctypes.c_int32), B, _ptr(k_new, ctypes.c_uint16),
                           _ptr(v_new, ctypes.c_uint16),
                           _ptr(q, ctypes.c_uint16) if q is not None else None,
                           num_q_heads, float(theta))
    _check(st, "oracle_append")
    return q


def decode_one(pool: np.ndarray, g: PoolGeom, bt_row, L: int, q_row, kv_head: int, scale: float,
               want_weights: bool = False):
    """One (sequence, query head): returns out[D] float64 (and weights[L])."""
    lib = _load()
    bt_row = _i32(bt_row)
    q_row = _u16(q_row)
    out = np.empty(g.head_dim, dtype=np.float64)
    w = np.empty(max(L, 1), dtype=np.float64) if want_weights else None
    st = lib.oracle_decode_one(_ptr(pool, ctypes.c_uint16), ctypes.byref(g), _ptr(bt_row, ctypes.c_int32),
                               bt_row.size, int(L), _ptr(q_row, ctypes.c_uint16), int(kv_head),
                               float(scale), _ptr(out, ctypes.c_double),
                               _ptr(w, ctypes.c_double) if w is not None else None)
    _check(st, "oracle_decode_one")
    return (out, w[:L]) if want_weights else out


def decode(pool: np.ndarray, g: PoolGeom, bt, seq_lens, q, scale: float):
    """Whole batch: returns (out_bf16 uint16 [B][Hq][D], out_f64 float64 [B][Hq][D])."""
    lib = _load()
    bt = _i32(bt)
    seq_lens = _i32(seq_lens)
    q = _u16(q)
    B, Hq, D = q.shape
    out_bf16 = np.empty((B, Hq, D), dtype=np.uint16)
    out_f64 = np.empty((B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode(_ptr(pool, ctypes.c_uint16), ctypes.byref(g), _ptr(bt, ctypes.c_int32),
                           bt.shape[1], _ptr(seq_lens, ctypes.c_int32), B, _ptr(q, ctypes.c_uint16), Hq,
                           float(scale), _ptr(out_bf16, ctypes.c_uint16), _ptr(out_f64, ctypes.c_double))
    _check(st, "oracle_decode")
    return out_bf16, out_f64


def decode_contiguous(K, V, seq_lens, q, scale: float) -> np.ndarray:
    """Brute force over a contiguous cache: K, V [B][Hkv][S][D], q [B][Hq][D] (float64)."""
    lib = _load()
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    seq_lens = _i32(seq_lens)
    B, Hkv, S, D = K.shape
    Hq = q.shape[1]
    out = np.empty((B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_contiguous(_ptr(K, ctypes.c_double), _ptr(V, ctypes.c_double), S,
                                      _ptr(seq_lens, ctypes.c_int32), B, _ptr(q, ctypes.c_double), Hq,
                                      Hkv, D, float(scale), _ptr(out, ctypes.c_double))
    _check(st, "oracle_decode_contiguous")
    return out


def library_path() -> str:
    return os.path.abspath(_build.LIB)


# --------------------------------------------------------------------------- FP8 KV pages

FP8_PAGE_BYTES = 2 * 8 * 16 * (64 + 4)   # codes + row scales, for 8 KV heads x 16 slots x 64 dims


def _load_fp8():
    lib = _load()
    if getattr(lib, "_fp8_bound", False):
        return lib
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    f32p = ctypes.POINTER(ctypes.c_float)
    gp = ctypes.POINTER(PoolGeom)
    lib.oracle_e4m3_from_double.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_quantize_row_fp8.argtypes = [u16p, ctypes.c_int, u8p, f32p]
    lib.oracle_quantize_row_fp8.restype = None
    lib.oracle_fp8_code_offset.argtypes = [gp] + [ctypes.c_int] * 5
    lib.oracle_fp8_code_offset.restype = ctypes.c_int64
    lib.oracle_fp8_scale_offset.argtypes = [gp] + [ctypes.c_int] * 4
    lib.oracle_fp8_scale_offset.restype = ctypes.c_int64
    lib.oracle_append_fp8.argtypes = [u8p, gp, i32p, ctypes.c_int, i32p, ctypes.c_int, u16p, u16p, u16p,
                                      ctypes.c_int, ctypes.c_double]
    lib.oracle_append_fp8.restype = ctypes.c_int
    lib.oracle_decode_one_fp8.argtypes = [u8p, gp, i32p, ctypes.c_int, ctypes.c_int, u16p, ctypes.c_int,
                                          ctypes.c_double, f64p, f64p]
    lib.oracle_decode_one_fp8.restype = ctypes.c_int
    lib.oracle_decode_fp8.argtypes = [u8p, gp, i32p, ctypes.c_int, i32p, ctypes.c_int, u16p, ctypes.c_int,
                                      ctypes.c_double, u16p, f64p]
    lib.oracle_decode_fp8.restype = ctypes.c_int
    lib._fp8_bound = True
    return lib


def e4m3_from_f64(values) -> np.ndarray:
    lib = _load_fp8()
    v = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
    return np.array([lib.oracle_e4m3_from_double(float(x)) for x in v], dtype=np.uint8).reshape(np.shape(values))


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load_fp8()
    c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib.oracle_e4m3_to_double(int(x)) for x in c], dtype=np.float64).reshape(np.shape(codes))


def quantize_row_fp8(row_bf16):
    """One row of BF16 bits -> (codes uint8, scale float32)."""
    lib = _load_fp8()
    row = _u16(row_bf16)
    codes = np.empty(row.size, dtype=np.uint8)
    scale = ctypes.c_float()
    lib.oracle_quantize_row_fp8(_ptr(row, ctypes.c_uint16), row.size, _ptr(codes, ctypes.c_uint8),
                                ctypes.byref(scale))
    return codes, np.float32(scale.value)


def fp8_code_offset(g: PoolGeom, page, kv, head, slot, dim) -> int:
    return int(_load_fp8().oracle_fp8_code_offset(ctypes.byref(g), page, kv, head, slot, dim))


def fp8_scale_offset(g: PoolGeom, page, kv, head, slot) -> int:
    return int(_load_fp8().oracle_fp8_scale_offset(ctypes.byref(g), page, kv, head, slot))


def append_fp8(pool: np.ndarray, g: PoolGeom, bt, pos, k_new, v_new, q=None, num_q_heads: int = 32,
               theta: float = 500000.0):
    """As ``append`` for an FP8 pool (uint8 bytes, modified in place)."""
    lib = _load_fp8()
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    bt, pos = _i32(bt), _i32(pos)
    k_new, v_new = _u16(k_new), _u16(v_new)
    B, max_blocks = bt.shape
    st = lib.oracle_append_fp8(_ptr(pool, ctypes.c_uint8), ctypes.byref(g), _ptr(bt, ctypes.c_int32), max_blocks,
                               _ptr(pos, ctypes.c_int32), B, _ptr(k_new, ctypes.c_uint16),
                               _ptr(v_new, ctypes.c_uint16), _ptr(q, ctypes.c_uint16) if q is not None else None,
                               num_q_heads, float(theta))
    _check(st, "oracle_append_fp8")
    return q


def decode_one_fp8(pool, g: PoolGeom, bt_row, L: int, q_row, kv_head: int, scale: float):
    lib = _load_fp8()
    bt_row, q_row = _i32(bt_row), _u16(q_row)
    out = np.empty(g.head_dim, dtype=np.float64)
    st = lib.oracle_decode_one_fp8(_ptr(pool, ctypes.c_uint8), ctypes.byref(g), _ptr(bt_row, ctypes.c_int32),
                                   bt_row.size, int(L), _ptr(q_row, ctypes.c_uint16), int(kv_head), float(scale),
                                   _ptr(out, ctypes.c_double), None)
    _check(st, "oracle_decode_one_fp8")
    return out


def decode_fp8(pool, g: PoolGeom, bt, seq_lens, q, scale: float):
    lib = _load_fp8()
    bt, seq_lens, q = _i32(bt), _i32(seq_lens), _u16(q)
    B, Hq, D = q.shape
    out_bf16 = np.empty((B, Hq, D), dtype=np.uint16)
    out_f64 = np.empty((B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_fp8(_ptr(pool, ctypes.c_uint8), ctypes.byref(g), _ptr(bt, ctypes.c_int32), bt.shape[1],
                               _ptr(seq_lens, ctypes.c_int32), B, _ptr(q, ctypes.c_uint16), Hq, float(scale),
                               _ptr(out_bf16, ctypes.c_uint16), _ptr(out_f64, ctypes.c_double))
    _check(st, "oracle_decode_fp8")
    return out_bf16, out_f64
