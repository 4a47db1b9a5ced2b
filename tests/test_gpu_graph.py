"""CUDA-graph capture of a step (write_slots + attention_varlen) through the
C ABI: the captured graph replays exactly what the eager calls compute, on
new inputs too, and a capture whose lengths were not prepared is refused."""
import numpy as np
import pytest
import torch

import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _batch(kind):
    if kind == "mixed":     # decodes and a prefill chunk: one mixed launch
        s = W.custom_spec("graph_mixed", 32, 8, 16, [1, 1, 130, 1], [500, 3000, 1200, 64], seed=11)
    elif kind == "nvfp4":   # NVFP4 pools: decodes and a chunked prefill
        s = W.custom_spec("graph_nvfp4", 32, 8, 16, [1, 1, 30, 1], [500, 3000, 1200, 64], seed=13,
                          kv_dtype="nvfp4")
    else:                   # decodes only
        s = W.custom_spec("graph_decode", 32, 8, 16, [1] * 6, [100, 5000, 20000, 17, 333, 4096], seed=12)
    return W.generate(s, DEV)


@pytest.mark.parametrize("kind", ["mixed", "decode", "nvfp4"])
def test_captured_step_replays_like_eager(kind):
    b = _batch(kind)
    h = U.make_handle(b, flags=pkv.FLAG_VALIDATE)
    m = U.device_meta(b)

    def step(out, lse):
        h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
        h.attention_varlen(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"],
                           b.qsl, b.seq_lens, out=out, lse=lse, k_scale=b.k_scale,
                           v_scale=b.v_scale)

    T, Hq = b.q.shape[0], b.q.shape[1]
    out_e = torch.empty_like(b.q)
    lse_e = torch.empty((T, Hq), dtype=torch.float32, device=DEV)
    out_g = torch.full_like(b.q, float("nan"))
    lse_g = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    step(out_e, lse_e)
    torch.cuda.synchronize()

    h.graph_prepare(b.qsl, b.seq_lens)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(out_g, lse_g)
    g.replay()
    torch.cuda.synchronize()
    h.check_device_errors()
    assert torch.equal(out_g, out_e) and torch.equal(lse_g, lse_e)

    # new queries and new K/V rows through the same graph
    gen = torch.Generator(device="cpu").manual_seed(99)
    b.q.copy_(torch.randn(b.q.shape, generator=gen).to(b.q.dtype))
    b.k_new.copy_(torch.randn(b.k_new.shape, generator=gen).to(b.k_new.dtype))
    g.replay()
    step(out_e, lse_e)
    torch.cuda.synchronize()
    h.check_device_errors()
    assert torch.equal(out_g, out_e) and torch.equal(lse_g, lse_e)
    sub = W.subset(b, list(range(b.spec.num_seqs)))
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    got, got_lse = U.gpu_rows(out_g, lse_g, sub)
    U.check(got, ref, got_lse, ref_lse, b.spec.kv_dtype, f"graph_{kind}", scaled=True)
    h.close()


def test_capture_without_matching_prepare_is_refused():
    b = _batch("decode")
    h = U.make_handle(b)
    m = U.device_meta(b)
    h.graph_prepare(b.qsl, b.seq_lens)
    other = b.seq_lens.copy()
    other[0] += 1
    out = torch.empty_like(b.q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        with pytest.raises(pkv.PkvError) as e:
            h.attention_varlen(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"],
                               b.qsl, other, out=out)
    assert "pkv_graph_prepare" in str(e.value)
    h.close()
