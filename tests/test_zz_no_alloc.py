"""pkv_decode_static, the decode entry point that allocates nothing.

It serves callers that cannot allocate GPU memory (their pool owns the whole
device, or they may not allocate after start-up), so its scratch is a fixed
array inside the library.  Checked on the GPU against pkv_attention_varlen,
through the C ABI, on two calls in a row (the second call reuses the array
the first one left behind).  Collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv,bs,hq,hkv,lens", [
    ("bf16", 16, 32, 8, [9000, 4097, 17, 30000, 1, 12345]),
    ("fp8", 64, 64, 8, [70000, 65, 3000]),
    ("nvfp4", 16, 32, 8, [20000, 33, 5000]),
])
def test_static_scratch_decode_matches_the_handle_path(kv, bs, hq, hkv, lens):
    s = W.custom_spec("static", hq, hkv, bs, [1] * len(lens), lens, seed=11, kv_dtype=kv)
    b = W.generate(s, "cuda")
    h = U.make_handle(b, flags=0)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    ref, ref_lse = h.attention_varlen(
        b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"], b.qsl, b.seq_lens,
        lse=torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda"),
        k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    h.close()
    for call in range(2):
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.decode_static(h.config, b.q, b.k_cache, b.v_cache, m["bt"], b.qsl,
                          b.seq_lens, out=out, lse=lse, k_scale=b.k_scale,
                          v_scale=b.v_scale)
        torch.cuda.synchronize()
        U.check(out.double().cpu().numpy().reshape(-1, 128),
                ref.double().cpu().numpy().reshape(-1, 128),
                lse.double().cpu().numpy().reshape(-1),
                ref_lse.double().cpu().numpy().reshape(-1), kv, f"static call {call}")


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
