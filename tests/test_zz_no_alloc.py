"""pkv_decode_static, the decode entry point that allocates nothing.

It serves callers that cannot allocate GPU memory (their memory pool owns the
whole device, or they may not allocate after start-up), so its scratch is a
fixed array inside the library.  Checked on the GPU through the C ABI: on two
calls in a row (the second reuses the array the first one left behind)
against pkv_attention_varlen and, for one case, against the oracle; free
device memory does not move across a call; a bad block id comes back through
pkv_decode_static_errors.  Collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _batch(kv, bs, hq, hkv, lens, seed=11):
    s = W.custom_spec("static", hq, hkv, bs, [1] * len(lens), lens, seed=seed, kv_dtype=kv)
    return W.generate(s, "cuda")


@pytest.mark.parametrize("kv,bs,hq,hkv,lens", [
    ("bf16", 16, 32, 8, [9000, 4097, 17, 30000, 1, 12345]),
    ("fp8", 64, 64, 8, [70000, 65, 3000]),
    ("nvfp4", 16, 32, 8, [20000, 33, 5000]),
])
def test_static_scratch_decode_matches_the_handle_path(kv, bs, hq, hkv, lens):
    b = _batch(kv, bs, hq, hkv, lens)
    h = U.make_handle(b, flags=0)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    ref, ref_lse = h.attention_varlen(
        b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"], b.qsl, b.seq_lens,
        lse=torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda"),
        k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    cfg = h.config
    h.close()
    pkv.decode_static_setup(cfg)                # the one-time set-up (warm-up)
    outs = [torch.full_like(b.q, float("nan")) for _ in range(2)]
    lses = [torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
            for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):
        free0 = torch.cuda.mem_get_info()[0]
        pkv.decode_static(cfg, b.q, b.k_cache, b.v_cache, m["bt"], b.qsl, b.seq_lens,
                          out=outs[call], lse=lses[call], k_scale=b.k_scale,
                          v_scale=b.v_scale)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "the call changed free device memory"
        U.check(outs[call].double().cpu().numpy().reshape(-1, 128),
                ref.double().cpu().numpy().reshape(-1, 128),
                lses[call].double().cpu().numpy().reshape(-1),
                ref_lse.double().cpu().numpy().reshape(-1), kv, f"static call {call}",
                scaled=True)
    pkv.decode_static_errors()


def test_static_scratch_decode_matches_the_oracle():
    """One bf16 batch (split and unsplit requests) against the fp64 oracle,
    every row, on two calls in a row."""
    b = _batch("bf16", 16, 32, 8, [20000, 4097, 17, 1], seed=13)
    sub = W.subset(b, list(range(b.spec.num_seqs)))      # pools before the append
    h = U.make_handle(b, flags=0)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache)
    torch.cuda.synchronize()
    cfg = h.config
    h.close()
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    for call in range(2):
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.decode_static(cfg, b.q, b.k_cache, b.v_cache, m["bt"], b.qsl, b.seq_lens,
                          out=out, lse=lse)
        torch.cuda.synchronize()
        got, got_lse = U.gpu_rows(out, lse, sub)
        U.check(got, ref, got_lse, ref_lse, "bf16", f"static vs oracle, call {call}",
                scaled=True)
    pkv.decode_static_errors()


def test_static_scratch_reports_bad_block_ids():
    """A block-table entry outside the pool is read as zeros (TMA fills rows
    outside its map) and recorded; pkv_decode_static_errors reports it once
    and clears it."""
    b = _batch("bf16", 16, 8, 2, [100, 60])
    m = U.device_meta(b)
    cfg = pkv.make_config(8, 2, 16, b.num_blocks, 2, 2)
    pkv.decode_static_setup(cfg)
    pkv.decode_static_errors()
    bad = m["bt"].clone()
    bad[0, 1] = b.num_blocks + 5
    out = torch.empty_like(b.q)
    pkv.decode_static(cfg, b.q, b.k_cache, b.v_cache, bad, b.qsl, b.seq_lens, out=out)
    with pytest.raises(pkv.PkvError) as e:
        pkv.decode_static_errors()
    assert e.value.status == 5
    pkv.decode_static_errors()                  # cleared
    pkv.decode_static(cfg, b.q, b.k_cache, b.v_cache, m["bt"], b.qsl, b.seq_lens, out=out)
    pkv.decode_static_errors()                  # a clean call records nothing


def test_static_scratch_limits_are_reported():
    cfg = pkv.make_config(8, 8, 16, 1000, 1, 1)
    q = torch.zeros((2100, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1000, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((2100, 1), dtype=torch.int32, device="cuda")
    qsl = np.arange(2101, dtype=np.int32)
    lens = np.ones(2100, dtype=np.int32)
    with pytest.raises(pkv.PkvError) as e:      # 2100 requests x 8 KV heads
        pkv.decode_static(cfg, q, kc, kc, bt, qsl, lens)
    assert e.value.status == 7
    with pytest.raises(pkv.PkvError) as e:      # prefill rows are not served
        pkv.decode_static(cfg, q[:9], kc, kc, bt[:1], np.array([0, 9], np.int32),
                          np.array([9], np.int32))
    assert e.value.status == 2
