"""Python binding of libpkv: paged, prefix-cached KV attention on GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``libpkv.so`` behind the C ABI in ``include/pkv.h``; the names here
mirror those entry points.  PyTorch is used for device memory and streams.
If the library has not been built (``python -m
paged_kv_attention_pkv_gb300.build`` or ``__graft_entry__.build()``), loading
fails with an error: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_CUDA", 4: "PKV_ERR_OUT_OF_MEMORY",
                5: "PKV_ERR_DEVICE_CHECK", 6: "PKV_ERR_TIMEOUT",
                7: "PKV_ERR_WORKSPACE"}
KV_BF16, KV_FP8_E4M3, KV_NVFP4 = 0, 1, 2
FLAG_VALIDATE, FLAG_TIMING, FLAG_SEPARATE = 1, 2, 4
KERNEL_APPEND, KERNEL_DECODE, KERNEL_PREFILL, KERNEL_MIXED, KERNEL_MERGE, KERNEL_STAGE = \
    0, 1, 2, 3, 4, 5

# Every symbol include/pkv.h declares.
EXPORTS = ["pkv_create", "pkv_write_slots", "pkv_attention_varlen",
           "pkv_check_device_errors", "pkv_status_string", "pkv_last_error",
           "pkv_destroy", "pkv_plan", "pkv_timing_reset", "pkv_timing_read",
           "pkv_decode_static", "pkv_decode_static_errors", "pkv_wait_selftest",
           "pkv_graph_prepare",
           "pkv_attention_partial",
           "pkv_lse_merge", "pkv_rope_write_slots",
           # host block pool (include/pkv_blocks.h)
           "pkv_blocks_create", "pkv_blocks_destroy", "pkv_blocks_lookup",
           "pkv_blocks_allocate", "pkv_blocks_commit", "pkv_blocks_free",
           "pkv_blocks_slots", "pkv_blocks_stats", "pkv_blocks_ref_count"]


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("num_blocks", ctypes.c_int64), ("max_num_seqs", ctypes.c_int32),
                ("max_num_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("stage_tokens", ctypes.c_int64)]


class WorkItem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kind", "seq", "kv_head", "tok0", "row0", "n_rows", "hist",
                 "k_begin", "k_end", "part", "pair", "n_split")]


_lib = None


def load(path: str | None = None):
    """Load libpkv.so and declare its C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    so = path or LIB_PATH
    if not os.path.exists(so):
        raise RuntimeError(
            f"{so} is missing: build the CUDA library first "
            "(python -m paged_kv_attention_pkv_gb300.build)")
    lib = ctypes.CDLL(so)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.pkv_create.restype = ctypes.c_int
    lib.pkv_create.argtypes = [ctypes.POINTER(Config), ctypes.c_int, ctypes.POINTER(vp)]
    lib.pkv_write_slots.restype = ctypes.c_int
    lib.pkv_write_slots.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
    lib.pkv_attention_varlen.restype = ctypes.c_int
    lib.pkv_attention_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                         vp, vp, i32, i32, vp, vp, vp]
    lib.pkv_check_device_errors.restype = ctypes.c_int
    lib.pkv_check_device_errors.argtypes = [vp]
    lib.pkv_attention_partial.restype = ctypes.c_int
    lib.pkv_attention_partial.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                          vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.pkv_rope_write_slots.restype = ctypes.c_int
    lib.pkv_rope_write_slots.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, vp, i32, vp, vp,
                                         vp, vp, vp]
    lib.pkv_lse_merge.restype = ctypes.c_int
    lib.pkv_lse_merge.argtypes = [vp, vp, vp, i32, i64, vp, vp, vp]
    i64p = ctypes.POINTER(i64)
    for n, args in (("pkv_blocks_create", [i64, i32, ctypes.POINTER(vp)]),
                    ("pkv_blocks_destroy", [vp]),
                    ("pkv_blocks_lookup", [vp, vp, i64, i64p]),
                    ("pkv_blocks_allocate", [vp, i64, vp, i64, i64, i32, vp, i64, i64p, i64p,
                                             ctypes.POINTER(i32)]),
                    ("pkv_blocks_commit", [vp, i64, vp, i64, i64]),
                    ("pkv_blocks_free", [vp, i64]),
                    ("pkv_blocks_slots", [vp, i64, i64, i64, vp]),
                    ("pkv_blocks_stats", [vp, i64p, i64p, i64p]),
                    ("pkv_blocks_ref_count", [vp, i32])):
        getattr(lib, n).restype = ctypes.c_int32
        getattr(lib, n).argtypes = args
    lib.pkv_graph_prepare.restype = ctypes.c_int
    lib.pkv_graph_prepare.argtypes = [vp, vp, vp, i32, i32]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_last_error.argtypes = [vp]
    lib.pkv_destroy.restype = ctypes.c_int
    lib.pkv_destroy.argtypes = [vp]
    lib.pkv_plan.restype = ctypes.c_int
    lib.pkv_plan.argtypes = [ctypes.POINTER(Config), vp, vp, i32, i32, i32,
                             ctypes.POINTER(WorkItem), i32, ctypes.POINTER(i32),
                             ctypes.POINTER(i32)]
    lib.pkv_timing_reset.restype = ctypes.c_int
    lib.pkv_timing_reset.argtypes = [vp]
    lib.pkv_timing_read.restype = ctypes.c_int
    lib.pkv_timing_read.argtypes = [vp, i32, ctypes.POINTER(i32),
                                    ctypes.POINTER(ctypes.c_double)]
    lib.pkv_decode_static.restype = ctypes.c_int
    lib.pkv_decode_static.argtypes = [ctypes.POINTER(Config), vp, vp, vp, vp, vp, vp,
                                      i32, vp, vp, i32, i32, vp, vp, vp]
    lib.pkv_decode_static_errors.restype = ctypes.c_int
    lib.pkv_decode_static_errors.argtypes = [vp]
    lib.pkv_wait_selftest.restype = ctypes.c_int
    lib.pkv_wait_selftest.argtypes = [vp, ctypes.c_uint64, vp]
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def _ptr(x) -> ctypes.c_void_p | None:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return ctypes.c_void_p(x.data_ptr())
    if isinstance(x, np.ndarray):
        return ctypes.c_void_p(x.ctypes.data)
    return ctypes.c_void_p(int(x))


def _host_i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_config(num_q_heads, num_kv_heads, block_size, num_blocks, max_num_seqs,
                max_num_tokens, kv_dtype=KV_BF16, softmax_scale=None, flags=0,
                head_dim=128, stage_tokens=0) -> Config:
    if softmax_scale is None:
        softmax_scale = head_dim ** -0.5
    return Config(num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype,
                  float(softmax_scale), int(num_blocks), max_num_seqs,
                  max_num_tokens, flags, int(stage_tokens))


def pool_shapes(config: Config):
    """Shapes and dtypes of the K (and V) pool and of the block-scale arrays
    a handle with ``config`` reads: ``(pool_shape, pool_dtype, scale_shape)``,
    ``scale_shape`` None for bf16 pools.  bf16 and E4M3 pools are
    ``[num_blocks, Hkv, block_size, 128]`` (bf16 / uint8); NVFP4 pools are
    ``[num_blocks, Hkv, block_size * 72]`` uint8 (include/pkv.h, pool layout)."""
    nb, hkv, bs = int(config.num_blocks), int(config.num_kv_heads), int(config.block_size)
    if config.kv_dtype == KV_NVFP4:
        return (nb, hkv, bs * 72), torch.uint8, (nb, hkv)
    if config.kv_dtype == KV_FP8_E4M3:
        return (nb, hkv, bs, int(config.head_dim)), torch.uint8, (nb, hkv)
    return (nb, hkv, bs, int(config.head_dim)), torch.bfloat16, None


class Handle:
    """A libpkv handle bound to one CUDA device (pkv_create / pkv_destroy)."""

    def __init__(self, config: Config, device: int = 0):
        self._lib = load()
        self.config = config
        self.device = device
        h = ctypes.c_void_p()
        st = self._lib.pkv_create(ctypes.byref(config), device, ctypes.byref(h))
        if st != PKV_OK:
            raise PkvError(st, self._lib.pkv_last_error(None).decode())
        self._h = h

    def _check(self, st: int):
        if st != PKV_OK:
            raise PkvError(st, self._lib.pkv_last_error(self._h).decode())

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def fp8(self) -> bool:
        return self.config.kv_dtype == KV_FP8_E4M3

    def write_slots(self, k_new, v_new, slot_mapping, k_cache, v_cache,
                    k_scale=None, v_scale=None, stream=None) -> None:
        """pkv_write_slots: append this step's K/V rows at their slots."""
        self._check(self._lib.pkv_write_slots(
            self._h, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
            int(slot_mapping.shape[0]), _ptr(k_cache), _ptr(v_cache),
            _ptr(k_scale), _ptr(v_scale), _stream(stream, self.device)))

    def rope_write_slots(self, q, k_new, v_new, positions, cos_sin_cache, slot_mapping,
                         k_cache, v_cache, neox=True, k_scale=None, v_scale=None,
                         stream=None) -> None:
        """pkv_rope_write_slots: rotate q in place, rotate and append K, append V."""
        self._check(self._lib.pkv_rope_write_slots(
            self._h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(cos_sin_cache),
            int(cos_sin_cache.shape[0]), int(bool(neox)), _ptr(slot_mapping),
            int(slot_mapping.shape[0]), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
            _ptr(v_scale), _stream(stream, self.device)))

    def attention_varlen(self, q, k_cache, v_cache, query_start_loc, seq_lens,
                         block_tables, query_start_loc_host, seq_lens_host,
                         out=None, lse=None, k_scale=None, v_scale=None,
                         stream=None):
        """pkv_attention_varlen: one step over a mixed varlen batch.

        Returns ``(out, lse)``; ``out`` is allocated if not given.  ``lse``
        is written only when a tensor is passed.
        """
        qslh = _host_i32(query_start_loc_host)
        lenh = _host_i32(seq_lens_host)
        if out is None:
            out = torch.empty_like(q)
        self._check(self._lib.pkv_attention_varlen(
            self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
            _ptr(v_scale), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_tables),
            int(block_tables.shape[1]), _ptr(qslh), _ptr(lenh), int(lenh.shape[0]),
            int(q.shape[0]), _ptr(out), _ptr(lse), _stream(stream, self.device)))
        return out, lse

    def attention_partial(self, q, k_cache, v_cache, query_start_loc, seq_lens,
                          block_tables, query_start_loc_host, seq_lens_host, shard,
                          num_shards, interleave, out=None, lse=None, k_scale=None,
                          v_scale=None, stream=None):
        """pkv_attention_partial: one context-parallel shard's partial output
        (fp32, ``[T, Hq, 128]``) and log-sum-exp (``[T, Hq]``)."""
        qslh = _host_i32(query_start_loc_host)
        lenh = _host_i32(seq_lens_host)
        T, hq = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty((T, hq, q.shape[2]), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
        self._check(self._lib.pkv_attention_partial(
            self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
            _ptr(v_scale), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_tables),
            int(block_tables.shape[1]), _ptr(qslh), _ptr(lenh), int(lenh.shape[0]),
            int(T), int(shard), int(num_shards), int(interleave), _ptr(out), _ptr(lse),
            _stream(stream, self.device)))
        return out, lse

    def lse_merge(self, parts_o, parts_lse, out=None, lse=None, stream=None):
        """pkv_lse_merge: ``parts_o`` ``[N, rows..., 128]`` fp32 and
        ``parts_lse`` ``[N, rows...]`` fp32 -> bf16 ``out`` ``[rows..., 128]``
        (and ``lse`` if given)."""
        n = parts_o.shape[0]
        rows = parts_lse[0].numel()
        if out is None:
            out = torch.empty(parts_o.shape[1:], dtype=torch.bfloat16, device=parts_o.device)
        self._check(self._lib.pkv_lse_merge(self._h, _ptr(parts_o), _ptr(parts_lse), int(n),
                                            int(rows), _ptr(out), _ptr(lse),
                                            _stream(stream, self.device)))
        return out, lse

    def graph_prepare(self, query_start_loc_host, seq_lens_host, num_tokens=None) -> None:
        """pkv_graph_prepare: plan a step for CUDA-graph capture (synchronous;
        call before capturing attention_varlen with the same host mirrors)."""
        qslh = _host_i32(query_start_loc_host)
        lenh = _host_i32(seq_lens_host)
        nt = int(qslh[-1]) if num_tokens is None else int(num_tokens)
        self._check(self._lib.pkv_graph_prepare(self._h, _ptr(qslh), _ptr(lenh),
                                                int(lenh.shape[0]), nt))

    def check_device_errors(self) -> None:
        """pkv_check_device_errors: raise PkvError if the device recorded one."""
        self._check(self._lib.pkv_check_device_errors(self._h))

    def wait_selftest(self, limit_ns: int, stream=None) -> None:
        """pkv_wait_selftest: one bounded wait that runs out after limit_ns;
        the next check_device_errors reports the timeout."""
        self._check(self._lib.pkv_wait_selftest(self._h, int(limit_ns),
                                                _stream(stream, self.device)))

    def timing_reset(self) -> None:
        self._check(self._lib.pkv_timing_reset(self._h))

    def timing_read(self, kind: int) -> tuple[int, float]:
        """(launches, total milliseconds) of one kernel kind since the reset."""
        n = ctypes.c_int32()
        ms = ctypes.c_double()
        self._check(self._lib.pkv_timing_read(self._h, kind, ctypes.byref(n),
                                              ctypes.byref(ms)))
        return n.value, ms.value


class Blocks:
    """Host block pool with prefix caching (include/pkv_blocks.h)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load()
        self.block_size = block_size
        h = ctypes.c_void_p()
        st = self._lib.pkv_blocks_create(num_blocks, block_size, ctypes.byref(h))
        if st != 0:
            raise PkvError(st, "pkv_blocks_create rejected its arguments")
        self._h = h

    def _call(self, name, *args):
        st = getattr(self._lib, name)(self._h, *args)
        if st != 0:
            raise PkvError(st, f"{name} rejected its arguments")

    def lookup(self, tokens) -> int:
        t = _host_i32(tokens)
        hit = ctypes.c_int64()
        self._call("pkv_blocks_lookup", _ptr(t), int(t.shape[0]), ctypes.byref(hit))
        return hit.value

    def allocate(self, req: int, tokens, num_new_tokens: int, num_lookahead: int = 0):
        """(block table or None if the pool cannot hold it, num_computed)."""
        t = _host_i32(tokens)
        cap = (int(t.shape[0]) + num_lookahead + self.block_size) // self.block_size + 1
        table = np.zeros(max(cap, 1), np.int32)
        nb, nc, ok = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        self._call("pkv_blocks_allocate", int(req), _ptr(t), int(t.shape[0]),
                   int(num_new_tokens), int(num_lookahead), _ptr(table), int(table.shape[0]),
                   ctypes.byref(nb), ctypes.byref(nc), ctypes.byref(ok))
        if not ok.value:
            return None, None
        return table[:nb.value].copy(), nc.value

    def commit(self, req: int, tokens, num_computed: int) -> None:
        t = _host_i32(tokens)
        self._call("pkv_blocks_commit", int(req), _ptr(t), int(t.shape[0]), int(num_computed))

    def free(self, req: int) -> None:
        self._call("pkv_blocks_free", int(req))

    def slots(self, req: int, pos0: int, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), np.int64)
        self._call("pkv_blocks_slots", int(req), int(pos0), int(n), _ptr(out))
        return out[:n]

    def stats(self) -> dict:
        f, c, e = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        self._call("pkv_blocks_stats", ctypes.byref(f), ctypes.byref(c), ctypes.byref(e))
        return {"free": f.value, "cached": c.value, "evictable": e.value}

    def ref_count(self, block: int) -> int:
        return self._lib.pkv_blocks_ref_count(self._h, int(block))

    def close(self) -> None:
        if self._h:
            self._lib.pkv_blocks_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan(config: Config, query_start_loc_host, seq_lens_host, num_sms: int = 152):
    """pkv_plan: the work items a step would run, as a list of dicts."""
    lib = load()
    qslh = _host_i32(query_start_loc_host)
    lenh = _host_i32(seq_lens_host)
    n = ctypes.c_int32()
    parts = ctypes.c_int32()
    st = lib.pkv_plan(ctypes.byref(config), _ptr(qslh), _ptr(lenh), int(lenh.shape[0]),
                      int(qslh[-1]) if qslh.size else 0, num_sms, None, 0,
                      ctypes.byref(n), ctypes.byref(parts))
    if st != PKV_OK:
        raise PkvError(st, lib.pkv_last_error(None).decode())
    arr = (WorkItem * max(n.value, 1))()
    st = lib.pkv_plan(ctypes.byref(config), _ptr(qslh), _ptr(lenh), int(lenh.shape[0]),
                      int(qslh[-1]), num_sms, arr, n.value, ctypes.byref(n),
                      ctypes.byref(parts))
    if st != PKV_OK:
        raise PkvError(st, lib.pkv_last_error(None).decode())
    items = [{f: getattr(arr[i], f) for f, _ in WorkItem._fields_} for i in range(n.value)]
    return items, parts.value


def decode_static(config: Config, q, k_cache, v_cache, block_tables,
                  query_start_loc_host, seq_lens_host, out=None, lse=None,
                  k_scale=None, v_scale=None, stream=None):
    """pkv_decode_static: split-KV decode on the current device with no
    handle and no allocation inside the library (its scratch is a fixed
    array compiled into libpkv).  For callers that cannot allocate GPU memory
    themselves; ``out`` must then be passed in.  Returns ``(out, lse)``."""
    lib = load()
    qslh = _host_i32(query_start_loc_host)
    lenh = _host_i32(seq_lens_host)
    if out is None:
        out = torch.empty_like(q)
    st = lib.pkv_decode_static(
        ctypes.byref(config), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), int(block_tables.shape[1]), _ptr(qslh),
        _ptr(lenh), int(lenh.shape[0]), int(q.shape[0]), _ptr(out), _ptr(lse),
        _stream(stream, q.device))
    if st != PKV_OK:
        raise PkvError(st, status_string(st))
    return out, lse


def decode_static_setup(config: Config) -> None:
    """pkv_decode_static with no requests: the one-time set-up on the current
    device (module load, kernel limits, error word cleared)."""
    st = load().pkv_decode_static(ctypes.byref(config), None, None, None, None, None,
                                  None, 0, None, None, 0, 0, None, None, None)
    if st != PKV_OK:
        raise PkvError(st, status_string(st))


def decode_static_errors(stream=None, device=None) -> None:
    """pkv_decode_static_errors: raise PkvError if the error word of the
    allocation-free decode holds anything (then cleared)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    st = load().pkv_decode_static_errors(_stream(stream, dev))
    if st != PKV_OK:
        raise PkvError(st, status_string(st))
