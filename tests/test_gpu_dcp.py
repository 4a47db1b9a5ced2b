"""Decode context parallelism emulated on one GPU, through the C ABI: each
shard's partial (pkv_attention_partial) against the oracle's shard partial,
and the merge of all shards (pkv_lse_merge) against the unsharded oracle and
the unsharded kernel."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # name, hq, hkv, bs, q_lens, seq_lens, kv, shards, interleave
    ("bf16_g4_n2_i16", 32, 8, 16, [1, 2, 1, 1], [5000, 777, 40, 1], "bf16", 2, 16),
    ("bf16_g4_n3_i256", 32, 8, 16, [1, 1, 2], [9000, 300, 2000], "bf16", 3, 256),
    ("bf16_g8_n2_i64", 64, 8, 64, [1, 1], [3000, 65], "bf16", 2, 64),
    ("bf16_g4_n1", 32, 8, 16, [1, 1], [1234, 17], "bf16", 1, 16),
    ("fp8_g8_n2_i64", 64, 8, 64, [1, 1, 1], [4000, 64, 129], "fp8", 2, 64),
    ("nvfp4_g8_n2_i64", 64, 8, 64, [1, 1, 1], [4000, 64, 129], "nvfp4", 2, 64),
    ("nvfp4_g4_n3_i128", 32, 8, 16, [1, 1], [5000, 300], "nvfp4", 3, 128),
    # the pages' interleave of 1 (token i on rank i % N), and runs shorter
    # than a decode stage: each shard walks the whole context, masking the
    # keys it does not own
    ("bf16_g4_n2_i1", 32, 8, 16, [1, 2, 1, 1], [5000, 777, 40, 1], "bf16", 2, 1),
    ("bf16_g4_n4_i1", 32, 8, 16, [1, 1, 2], [9000, 3, 2000], "bf16", 4, 1),
    ("bf16_g8_n8_i1", 64, 8, 64, [1, 1, 1], [3000, 65, 7], "bf16", 8, 1),
    ("fp8_g8_n2_i1", 64, 8, 64, [1, 1, 1], [4000, 64, 129], "fp8", 2, 1),
    ("fp8_g4_n4_i1", 32, 8, 16, [1, 1], [6000, 5], "fp8", 4, 1),
    ("fp8_g8_n8_i1", 64, 8, 64, [1, 1, 1], [20000, 33, 300], "fp8", 8, 1),
    ("nvfp4_g8_n4_i1", 64, 8, 64, [1, 1], [7000, 130], "nvfp4", 4, 1),
    ("bf16_g4_n3_i5", 32, 8, 16, [1, 1], [4000, 12], "bf16", 3, 5),
    ("fp8_g4_n2_i24", 32, 8, 16, [1, 2], [3000, 100], "fp8", 2, 24),
]


def _run(case):
    name, hq, hkv, bs, ql, sl, kv, n, k = case
    b = W.generate(W.custom_spec(name, hq, hkv, bs, ql, sl, seed=21, kv_dtype=kv), DEV)
    h = U.make_handle(b)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    parts = []
    for r in range(n):
        o, l = h.attention_partial(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"],
                                   b.qsl, b.seq_lens, r, n, k,
                                   k_scale=b.k_scale, v_scale=b.v_scale)
        parts.append((o, l))
    torch.cuda.synchronize()
    h.check_device_errors()
    return b, h, m, parts


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_shard_partials_match_the_oracle(case):
    name, hq, hkv, bs, ql, sl, kv, n, k = case
    b, h, m, parts = _run(case)
    sub = W.subset(b, list(range(b.spec.num_seqs)))
    kc, vc = sub["k_cache"].copy(), sub["v_cache"].copy()
    ks, vs = sub.get("k_scale"), sub.get("v_scale")
    oracle.write_slots(kc, vc, sub["k_new"], sub["v_new"], sub["slot_mapping"],
                       k_scale=ks, v_scale=vs)
    tol = U.TOL[kv]
    for r, (o, l) in enumerate(parts):
        ref, ref_lse = oracle.attention(kc, vc, sub["q"], sub["qsl"], sub["seq_lens"],
                                        sub["block_tables"], b.spec.softmax_scale,
                                        k_scale=ks, v_scale=vs, shard=(n, r, k))
        got, got_lse = U.gpu_rows(o, l, sub)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(got_lse), fin), f"{name} shard {r}: -inf rows differ"
        assert np.all(got[~fin] == 0.0)
        err = np.abs(got[fin] - ref[fin])
        assert err.max() <= tol["max_abs"], f"{name} shard {r}: max-abs {err.max():.3e}"
        assert err.mean() <= tol["mean_abs"], f"{name} shard {r}: mean-abs {err.mean():.3e}"
        assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= tol["lse"]
    h.close()


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_merged_shards_equal_the_unsharded_step(case):
    name, hq, hkv, bs, ql, sl, kv, n, k = case
    b, h, m, parts = _run(case)
    po = torch.stack([p[0] for p in parts])
    pl = torch.stack([p[1] for p in parts])
    lse = torch.empty_like(pl[0])
    out, _ = h.lse_merge(po, pl, lse=lse)
    full = torch.empty_like(b.q)
    full_lse = torch.empty_like(lse)
    h.attention_varlen(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"], b.qsl,
                       b.seq_lens, out=full, lse=full_lse, k_scale=b.k_scale,
                       v_scale=b.v_scale)
    torch.cuda.synchronize()
    sub = W.subset(b, list(range(b.spec.num_seqs)))
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    got, got_lse = U.gpu_rows(out, lse, sub)
    U.check(got, ref, got_lse, ref_lse, kv, f"{name} merged", scaled=True)
    if n == 1:
        # one shard is the unsharded plan: same fp32 result before rounding
        assert torch.equal(parts[0][0].to(torch.bfloat16), full)
        assert torch.equal(parts[0][1], full_lse)
    else:
        assert (out.float() - full.float()).abs().max().item() <= 2 * U.TOL[kv]["max_abs"]
    h.close()


def test_partial_refuses_prefill_rows_and_bad_arguments():
    b = W.generate(W.custom_spec("dcp_bad", 32, 8, 16, [1, 40], [100, 200], seed=3), DEV)
    h = U.make_handle(b)
    m = U.device_meta(b)
    args = (b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"], b.qsl, b.seq_lens)
    with pytest.raises(pkv.PkvError) as e:
        h.attention_partial(*args, 0, 2, 16)
    assert "decode rows" in str(e.value)
    b2 = W.generate(W.custom_spec("dcp_bad2", 32, 8, 16, [1, 1], [100, 200], seed=3), DEV)
    h2 = U.make_handle(b2)
    m2 = U.device_meta(b2)
    args2 = (b2.q, b2.k_cache, b2.v_cache, m2["qsl"], m2["lens"], m2["bt"], b2.qsl, b2.seq_lens)
    with pytest.raises(pkv.PkvError) as e:
        h2.attention_partial(*args2, 0, 2, 0)
    assert e.value.status == 1 and "interleave" in str(e.value)
    with pytest.raises(pkv.PkvError):
        h2.attention_partial(*args2, 2, 2, 16)
    h.close()
    h2.close()
