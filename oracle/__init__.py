"""fp64 CPU oracle for paged, prefix-cached KV attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it: the two share no code.  ``pkv_oracle.c``
states what is computed and which page and section each step follows.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force against a library attention routine, closed forms, invariances,
the FP8 format definition and a library FP8 cast, the FP4 format's published
value table and brute-force nearest rounding) and by
``tests/test_oracle_mutations.py`` (planted mistakes must fail those pins).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, library_path

_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    so = path or library_path()
    if path is None and not os.path.exists(so):
        build_oracle()
    lib = ctypes.CDLL(so)
    lib.pko_bf16_value.restype = ctypes.c_double
    lib.pko_bf16_value.argtypes = [ctypes.c_uint16]
    lib.pko_e4m3_value.restype = ctypes.c_double
    lib.pko_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.pko_e4m3_encode.restype = ctypes.c_uint8
    lib.pko_e4m3_encode.argtypes = [ctypes.c_float]
    lib.pko_e4m3_quantize.restype = ctypes.c_uint8
    lib.pko_e4m3_quantize.argtypes = [ctypes.c_uint16, ctypes.c_float]
    lib.pko_e2m1_value.restype = ctypes.c_double
    lib.pko_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.pko_e2m1_encode.restype = ctypes.c_uint8
    lib.pko_e2m1_encode.argtypes = [ctypes.c_float]
    lib.pko_nvfp4_quantize_row.restype = None
    lib.pko_nvfp4_quantize_row.argtypes = [_u16p, ctypes.c_int, ctypes.c_float,
                                           ctypes.c_void_p, ctypes.c_void_p]
    lib.pko_write_slots.restype = ctypes.c_int
    lib.pko_write_slots.argtypes = [
        ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int64, _u16p, _u16p, _i64p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p]
    lib.pko_attention.restype = ctypes.c_int
    lib.pko_attention.argtypes = [
        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, _u16p, _i32p, _i32p, _i32p, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int64, ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64, _f64p, _f64p]
    lib.pko_lse_merge.restype = None
    lib.pko_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p,
                                  _f64p, _f64p]
    lib.pko_bf16_round.restype = ctypes.c_uint16
    lib.pko_bf16_round.argtypes = [ctypes.c_double]
    lib.pko_rope.restype = ctypes.c_int
    lib.pko_rope.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _u16p, _i64p,
                             ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_void_p]
    lib.pko_num_threads.restype = ctypes.c_int
    lib.pko_num_threads.argtypes = []
    if path is None:
        _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(load().pko_num_threads())


def bf16_round(v: float, lib=None) -> int:
    """bf16 bit pattern of v rounded to nearest, ties to even."""
    return int((lib or load()).pko_bf16_round(float(v)))


def rope(x: np.ndarray, positions: np.ndarray, cos_sin: np.ndarray, neox: bool = True,
         lib=None):
    """Rotary embedding of ``x`` ``[T, H, d]`` (bf16 bits) at ``positions``
    with the ``[max_pos, d]`` fp32 cos/sin table; returns (fp64 values,
    bf16 bits), both ``[T, H, d]``."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    t, h, d = x.shape
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    f64 = np.zeros((t, h, d), np.float64)
    bits = np.zeros((t, h, d), np.uint16)
    st = lib.pko_rope(t, h, d, x, pos, _ptr(cs), cs.shape[0], int(bool(neox)), _ptr(f64),
                      _ptr(bits))
    if st != 0:
        raise ValueError(f"oracle rope rejected its arguments ({st})")
    return f64, bits


def bf16_value(bits: int) -> float:
    return float(load().pko_bf16_value(bits))


def e4m3_value(code: int) -> float:
    return float(load().pko_e4m3_value(code))


def e4m3_encode(x: float) -> int:
    return int(load().pko_e4m3_encode(x))


def e4m3_quantize(x_bf16_bits: int, scale: float) -> int:
    return int(load().pko_e4m3_quantize(x_bf16_bits, scale))


def e2m1_value(code: int) -> float:
    return float(load().pko_e2m1_value(code))


def e2m1_encode(x: float) -> int:
    return int(load().pko_e2m1_encode(x))


def nvfp4_quantize_row(x_bf16_bits: np.ndarray, scale: float):
    """NVFP4 codes (``d/2`` bytes) and E4M3 micro scales (``d/16``) of one
    row of bf16 bits under the (block, KV head) scale."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    d = x.shape[0]
    codes = np.zeros(d // 2, np.uint8)
    ms = np.zeros(d // 16, np.uint8)
    load().pko_nvfp4_quantize_row(x, d, float(scale), _ptr(codes), _ptr(ms))
    return codes, ms


def _pool_format(cache: np.ndarray, d: int | None = None):
    """(kv_fmt, num_blocks, hkv, bs, d) of a pool array: bf16 bits
    [nb, hkv, bs, d] uint16, E4M3 codes [nb, hkv, bs, d] uint8, or NVFP4
    tiles [nb, hkv, bs * 9 d / 16] uint8 (d = 128 unless given)."""
    if cache.ndim == 3:
        assert cache.dtype == np.uint8
        d = d or 128
        nb, hkv, tile = cache.shape
        assert tile % (9 * d // 16) == 0
        return 2, nb, hkv, tile // (9 * d // 16), d
    nb, hkv, bs, dd = cache.shape
    return (1 if cache.dtype == np.uint8 else 0), nb, hkv, bs, dd


def write_slots(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                v_new: np.ndarray, slot_mapping: np.ndarray,
                k_scale: np.ndarray | None = None,
                v_scale: np.ndarray | None = None, lib=None) -> None:
    """Scatter new K/V rows into the pools in place.

    Pools are ``[num_blocks, Hkv, bs, D]`` arrays of uint16 (bf16 bits) or
    uint8 (E4M3 codes), or ``[num_blocks, Hkv, bs * 9 D / 16]`` uint8 NVFP4
    tiles; quantised pools come with ``[num_blocks, Hkv]`` float32 scales.
    ``k_new`` and ``v_new`` are ``[T, Hkv, D]`` uint16 bf16 bits.
    """
    lib = lib or load()
    fmt, nb, hkv, bs, d = _pool_format(k_cache, k_new.shape[-1])
    quantised = fmt != 0
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    st = lib.pko_write_slots(
        fmt, int(k_new.shape[0]), hkv, d, bs, nb,
        np.ascontiguousarray(k_new), np.ascontiguousarray(v_new),
        np.ascontiguousarray(slot_mapping, dtype=np.int64),
        _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale) if quantised else None, _ptr(v_scale) if quantised else None)
    if st != 0:
        raise ValueError(f"oracle write_slots rejected its arguments ({st})")


def attention(k_cache: np.ndarray, v_cache: np.ndarray, q: np.ndarray,
              qsl: np.ndarray, seq_lens: np.ndarray, block_tables: np.ndarray,
              softmax_scale: float, k_scale: np.ndarray | None = None,
              v_scale: np.ndarray | None = None, rows: np.ndarray | None = None,
              k_range: tuple[int, int] | None = None,
              shard: tuple[int, int, int] | None = None, lib=None):
    """Paged varlen attention in fp64.

    ``q`` is ``[T, Hq, D]`` uint16 (bf16 bits).  Returns ``(out, lse)``:
    ``out`` is ``[nrows, D]`` float64 and ``lse`` ``[nrows]`` float64, where
    the rows are ``rows`` (indices ``token * Hq + head``) or all ``T * Hq``.
    ``k_range`` restricts keys to logical positions ``[lo, hi)``; ``shard =
    (n, r, k)`` to the keys context-parallel rank ``r`` of ``n`` owns when
    tokens are dealt out in runs of ``k`` (run ``j`` to rank ``j % n``).
    """
    lib = lib or load()
    t, hq, dq = q.shape
    fmt, nb, hkv, bs, d = _pool_format(k_cache, dq)
    quantised = fmt != 0
    assert dq == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    assert bt.ndim == 2
    qsl = np.ascontiguousarray(qsl, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
    nrows = t * hq if rows is None else rows.shape[0]
    out = np.zeros((nrows, d), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    lo, hi = (0, np.iinfo(np.int64).max) if k_range is None else k_range
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32) if quantised else None
    vs = np.ascontiguousarray(v_scale, dtype=np.float32) if quantised else None
    st = lib.pko_attention(
        fmt, _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs), nb, hkv, d,
        bs, hq, np.ascontiguousarray(q), qsl, seq_lens, bt, bt.shape[1],
        int(seq_lens.shape[0]), t, float(softmax_scale), int(lo), int(hi),
        *((1, 0, 1) if shard is None else tuple(int(x) for x in shard)),
        _ptr(rows), nrows, out, lse)
    if st != 0:
        raise ValueError(f"oracle attention rejected its arguments ({st})")
    return out, lse


def lse_merge(lse_parts: np.ndarray, o_parts: np.ndarray, lib=None):
    """Merge partial (o, lse) pairs over disjoint key sets into one."""
    lib = lib or load()
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.zeros((d,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    lib.pko_lse_merge(n, d, lse_parts, o_parts, o, lse)
    return o, float(lse[0])
