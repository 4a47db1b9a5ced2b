"""The C ABI: libpkv loads, exports every symbol include/*.h declares, and
rejects bad arguments with status codes (CPU only: no kernel is launched)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import paged_kv_attention_pkv_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                  if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("pkv_create", "pkv_write_slots", "pkv_attention_varlen", "pkv_destroy"):
        assert n in names
    assert names == sorted(pkv.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = pkv.load()
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_status_strings():
    for code in range(8):
        s = pkv.status_string(code)
        assert s and s != "unknown status"
    assert pkv.status_string(99) == "unknown status"


def test_null_handles_are_safe():
    lib = pkv.load()
    assert lib.pkv_destroy(None) == 0
    assert lib.pkv_timing_reset(None) == 0
    assert lib.pkv_check_device_errors(None) == 1
    assert lib.pkv_wait_selftest(None, 1000, None) == 1
    assert lib.pkv_write_slots(None, None, None, None, 0, None, None, None, None, None) == 1


def _cfg(**kw):
    base = dict(num_q_heads=32, num_kv_heads=8, block_size=16, num_blocks=1000,
                max_num_seqs=64, max_num_tokens=8192)
    base.update(kw)
    return pkv.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=30), 1), (dict(num_kv_heads=0), 1), (dict(num_blocks=0), 1),
    (dict(max_num_seqs=0), 1), (dict(softmax_scale=-1.0), 1), (dict(kv_dtype=7), 1),
    (dict(head_dim=64), 2), (dict(block_size=8), 2), (dict(block_size=48), 2),
    (dict(num_blocks=1 << 30), 2)])
def test_create_rejects_bad_config(kw, status):
    with pytest.raises(pkv.PkvError) as e:
        pkv.Handle(_cfg(**kw))
    assert e.value.status == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_create_without_gpu_reports_cuda_error():
    with pytest.raises(pkv.PkvError) as e:
        pkv.Handle(_cfg())
    assert e.value.status == 3


def test_pool_shapes_follow_the_header_layout():
    """bf16 / E4M3 pools are [num_blocks, Hkv, bs, 128]; NVFP4 pools hold 72
    bytes per token and KV head (64 code bytes + 8 micro scales)."""
    import torch
    for kv, shape, dtype, scales in (
            (pkv.KV_BF16, (10, 2, 16, 128), torch.bfloat16, None),
            (pkv.KV_FP8_E4M3, (10, 2, 16, 128), torch.uint8, (10, 2)),
            (pkv.KV_NVFP4, (10, 2, 16 * 72), torch.uint8, (10, 2))):
        cfg = pkv.make_config(8, 2, 16, 10, 4, 64, kv_dtype=kv)
        assert pkv.pool_shapes(cfg) == (shape, dtype, scales)
