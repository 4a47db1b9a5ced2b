"""CUDA path against the fp64 oracle, through the C ABI (GPU only).

Small cases compare every output row; the five workloads run at full size
and compare sampled rows the oracle computes one by one (always including
the first and last rows of each sequence and rows at tile boundaries).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = "cuda"


def spec(name, hq, hkv, bs, q_lens, seq_lens, kv="bf16", seed=7, shared=None):
    return W.custom_spec(name, hq, hkv, bs, q_lens, seq_lens, seed=seed,
                         kv_dtype=kv, shared_prefix=shared)


# ---- KV append -------------------------------------------------------------------

@pytest.mark.parametrize("kv,bs", [("bf16", 16), ("bf16", 64), ("fp8", 64), ("fp8", 16),
                                   ("nvfp4", 16), ("nvfp4", 64), ("nvfp4", 128)])
def test_write_slots_bit_exact(kv, bs):
    """Every byte of both pools equals the oracle's append (new rows at their
    slots, poison everywhere else), including -1 padding slots."""
    s = spec("append", 8, 2, bs, [3, 1, 40, 7], [50, 9, 140, 7], kv=kv)
    b = W.generate(s, DEV)
    b.slot_mapping[5] = -1                       # a padding token
    kc0, vc0 = W.host_pool(b, "k"), W.host_pool(b, "v")
    ks = b.k_scale.cpu().numpy() if b.k_scale is not None else None
    vs = b.v_scale.cpu().numpy() if b.v_scale is not None else None
    h = U.make_handle(b)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    torch.cuda.synchronize()
    h.check_device_errors()
    oracle.write_slots(kc0, vc0, W.bf16_bits(b.k_new), W.bf16_bits(b.v_new),
                       b.slot_mapping, k_scale=ks, v_scale=vs)
    assert np.array_equal(W.host_pool(b, "k"), kc0)
    assert np.array_equal(W.host_pool(b, "v"), vc0)


def test_write_slots_nvfp4_saturation_and_underflow_like_the_oracle():
    """NVFP4 append at the edges: K rows far above 6 * 448 * scale (micro
    scales saturate at 448, codes at 6) and V rows so small that micro
    scales round to 0 (all codes 0) or to E4M3 subnormals."""
    s = spec("sat4", 4, 2, 16, [5], [20], kv="nvfp4")
    b = W.generate(s, DEV)
    b.k_new.mul_(4000.0)
    b.v_new.mul_(1e-6)
    b.v_new[2].mul_(1e3)
    kc0, vc0 = W.host_pool(b, "k"), W.host_pool(b, "v")
    h = U.make_handle(b)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    torch.cuda.synchronize()
    oracle.write_slots(kc0, vc0, W.bf16_bits(b.k_new), W.bf16_bits(b.v_new),
                       b.slot_mapping, k_scale=b.k_scale.cpu().numpy(),
                       v_scale=b.v_scale.cpu().numpy())
    assert np.array_equal(W.host_pool(b, "k"), kc0)
    assert np.array_equal(W.host_pool(b, "v"), vc0)


def test_write_slots_fp8_saturates_like_the_oracle():
    """Values far beyond 448 * scale saturate to +-448 exactly as the oracle
    rounds them; ties and subnormal quotients round to nearest even."""
    s = spec("sat", 4, 2, 16, [4], [20], kv="fp8")
    b = W.generate(s, DEV)
    b.k_new.mul_(300.0)                          # push quotients past 448
    b.v_new.mul_(1e-4)                           # and into the subnormal range
    kc0, vc0 = W.host_pool(b, "k"), W.host_pool(b, "v")
    h = U.make_handle(b)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    torch.cuda.synchronize()
    oracle.write_slots(kc0, vc0, W.bf16_bits(b.k_new), W.bf16_bits(b.v_new),
                       b.slot_mapping, k_scale=b.k_scale.cpu().numpy(),
                       v_scale=b.v_scale.cpu().numpy())
    assert np.array_equal(W.host_pool(b, "k"), kc0)
    assert np.array_equal(W.host_pool(b, "v"), vc0)


# ---- small cases, every row -------------------------------------------------------

SWEEP = [
    # name, hq, hkv, bs, q_lens, seq_lens, kv
    ("mha_bs16", 8, 8, 16, [1, 2, 63, 64, 65, 129], [1, 17, 63, 80, 200, 129], "bf16"),
    ("gqa4_bs16", 32, 8, 16, [1, 2, 63, 64, 65, 129], [15, 16, 300, 64, 65, 1000], "bf16"),
    ("gqa8_bs64", 64, 8, 64, [1, 1, 2, 17, 1], [1, 64, 65, 1000, 4097], "bf16"),
    ("gqa2_bs32", 4, 2, 32, [3, 1, 31, 33], [3, 32, 95, 33], "bf16"),
    ("gqa4_bs128", 8, 2, 128, [2, 70], [129, 300], "bf16"),
    # query groups that are not powers of two: Q tiles of G * floor(128 / G) rows
    ("gqa3_tc", 6, 2, 16, [1, 2, 3, 40, 22, 130], [5, 100, 40, 300, 22, 900], "bf16"),
    ("gqa5_tc", 40, 8, 16, [1, 30, 51, 100], [70, 300, 51, 1000], "bf16"),
    ("gqa6_bs64", 48, 8, 64, [1, 43, 200], [1, 600, 2100], "bf16"),
    ("gqa12_tc", 96, 8, 16, [11, 25], [400, 25], "bf16"),
    ("gqa96_tc", 96, 1, 32, [1, 3, 5], [64, 700, 5], "bf16"),
    ("gqa16_tc", 32, 2, 16, [1, 9, 200], [300, 1000, 4000], "bf16"),
    ("fp8_gqa8_bs64", 64, 8, 64, [1, 1, 1, 1], [1, 63, 65, 5000], "fp8"),
    ("fp8_gqa4_bs16", 32, 8, 16, [1, 2, 1], [17, 33, 2000], "fp8"),
    # prefill rows without tensor-core tiles: 8-row chunks on the decode kernel
    ("fp8_prefill_gqa4", 32, 8, 16, [1, 40, 3, 130], [17, 300, 2000, 130], "fp8"),
    ("fp8_prefill_gqa8_bs64", 64, 8, 64, [1, 70, 5], [5000, 700, 65], "fp8"),
    ("fp8_prefill_gqa3", 6, 2, 64, [10, 1, 33], [100, 64, 1500], "fp8"),
    ("gqa256_chunks", 256, 1, 16, [1, 2, 9], [40, 50, 300], "bf16"),
    # NVFP4 pools (decode kernel; prefill rows as 8-row chunks)
    ("nvfp4_gqa8_bs64", 64, 8, 64, [1, 1, 1, 1], [1, 63, 65, 5000], "nvfp4"),
    ("nvfp4_gqa4_bs16", 32, 8, 16, [1, 2, 1, 40], [17, 33, 2000, 300], "nvfp4"),
    ("nvfp4_gqa2_bs128", 4, 2, 128, [1, 3, 1], [129, 700, 4100], "nvfp4"),
    ("nvfp4_gqa8_bs32", 16, 2, 32, [1, 1], [95, 3000], "nvfp4"),
    # NVFP4 prefill rows on the tensor cores (K and V converted to f16)
    ("nvfp4_prefill_gqa4", 32, 8, 16, [1, 40, 3, 130], [17, 300, 2000, 130], "nvfp4"),
    ("nvfp4_prefill_gqa8_bs64", 64, 8, 64, [1, 70, 5], [5000, 700, 65], "nvfp4"),
    ("nvfp4_prefill_gqa3", 6, 2, 64, [10, 1, 33], [100, 64, 1500], "nvfp4"),
    ("nvfp4_prefill_bs128", 16, 4, 128, [200, 2], [1300, 300], "nvfp4"),
    # quantised pools with query groups that leave TMEM lanes padded
    ("fp8_prefill_gqa12", 96, 8, 16, [11, 25], [400, 25], "fp8"),
    ("fp8_prefill_gqa96", 96, 1, 32, [1, 3, 5], [64, 700, 5], "fp8"),
    ("nvfp4_prefill_gqa12", 96, 8, 16, [11, 25], [400, 25], "nvfp4"),
    ("nvfp4_prefill_gqa96", 96, 1, 32, [1, 3, 5], [64, 700, 5], "nvfp4"),
    # few prefill tiles: key ranges split over the SMs, merged by the last
    # range to finish (boundaries at or below each tile's first position)
    ("split_q16_long", 32, 8, 16, [16], [8208], "bf16"),
    ("split_gqa3", 24, 8, 16, [300, 1], [2300, 900], "bf16"),
    ("split_bs256", 8, 2, 256, [33, 2], [3000, 700], "bf16"),
    ("split_fp8", 32, 8, 64, [40], [6000], "fp8"),
    ("split_nvfp4", 32, 8, 16, [40, 1], [6000, 3000], "nvfp4"),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: c[0])
@pytest.mark.parametrize("q_scale", [1.0, 8.0], ids=["normal", "peaked"])
def test_small_cases_every_row(case, q_scale):
    name, hq, hkv, bs, ql, sl, kv = case
    b = W.generate(spec(name, hq, hkv, bs, ql, sl, kv=kv), DEV, q_scale=q_scale)
    U.full_parity(b, what=name, peaked=q_scale > 1.0)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("separate", [False, True], ids=["one_launch", "separate"])
def test_mixed_step_launch_modes(separate, kv):
    """A step with decodes and prefill chunks runs as one mixed launch, or
    with PKV_FLAG_SEPARATE as a decode and a prefill launch; both match the
    oracle on every row.  E4M3 pools always take the two launches (measured
    faster there)."""
    s = spec("mixed_modes", 32, 4, 16, [1, 1, 300, 1, 77, 1], [40, 3000, 1300, 1, 77, 700],
             kv=kv)
    b = W.generate(s, DEV)
    flags = pkv.FLAG_VALIDATE | pkv.FLAG_TIMING | (pkv.FLAG_SEPARATE if separate else 0)
    h = U.make_handle(b, flags)
    sub = W.subset(b, list(range(s.num_seqs)))
    out, lse = U.gpu_step(b, handle=h)
    counts = {k: h.timing_read(k)[0] for k in
              (pkv.KERNEL_DECODE, pkv.KERNEL_PREFILL, pkv.KERNEL_MIXED)}
    h.close()
    ref, ref_lse = U.oracle_subset(sub, s)
    got, got_lse = U.gpu_rows(out, lse, sub)
    U.check(got, ref, got_lse, ref_lse, kv, f"mixed_modes {kv}")
    if separate or kv == "fp8":
        assert counts == {pkv.KERNEL_DECODE: 1, pkv.KERNEL_PREFILL: 1, pkv.KERNEL_MIXED: 0}
    else:
        assert counts == {pkv.KERNEL_DECODE: 0, pkv.KERNEL_PREFILL: 0, pkv.KERNEL_MIXED: 1}


def test_tiny_incremental_prefill_config():
    """1 sequence, l_hist 1000 + l_incr 64, 8q/2kv heads, 128-block pool."""
    b = W.generate(W.config_spec(0), DEV)
    U.full_parity(b, what="c1")


def test_prefix_shared_blocks():
    """Sessions sharing their first blocks read the same physical ids."""
    s = spec("shared", 32, 8, 16, [300, 40, 5, 1], [5000 + 300, 9000 + 40, 5000, 6000],
             shared=([0, 1, 2], 4800))
    b = W.generate(s, DEV)
    assert (b.block_tables[0, :300] == b.block_tables[1, :300]).all()
    U.full_parity(b, what="shared")


# ---- the five workloads at full size, sampled rows ---------------------------------

def _sampled(batch, seq_ids, kv_heads, token_pick=None, what=""):
    sub = W.subset(batch, seq_ids, kv_heads)
    hq = len(sub["heads"])
    rows = None
    if token_pick is not None:
        toks = []
        for r, i in enumerate(seq_ids):
            a = int(sub["qsl"][r])
            q = int(sub["qsl"][r + 1]) - a
            toks.extend(a + t for t in token_pick(q) if 0 <= t < q)
        toks = np.unique(np.asarray(toks, np.int64))
        rows = (toks[:, None] * hq + np.arange(hq)[None, :]).reshape(-1)
    out, lse = U.gpu_step(batch)
    ref, ref_lse = U.oracle_subset(sub, batch.spec, rows=rows)
    got, got_lse = U.gpu_rows(out, lse, sub, rows)
    return U.check(got, ref, got_lse, ref_lse, batch.spec.kv_dtype, what)


def _edge_tokens(q, G, rng=np.random.default_rng(3)):
    per_tile = max(1, 64 // G)
    picks = {0, 1, q - 2, q - 1, per_tile - 1, per_tile, 2 * per_tile}
    picks |= set(rng.integers(0, q, 6).tolist())
    return sorted(p for p in picks if 0 <= p < q)


def test_decode_batch_full_size():
    b = W.generate(W.config_spec(1), DEV)
    L = b.seq_lens
    seqs = sorted({int(L.argmin()), int(L.argmax()), 0, 17, 40, 63})
    _sampled(b, seqs, None, what="c2")


@pytest.mark.parametrize("kv", ["bf16", "fp8", "nvfp4"])
def test_post_tool_prefill_full_size(kv):
    """The post-tool-call prefill as bench.py times it (bf16, and the E4M3 /
    NVFP4 KV variants of its secondary lines): sessions 0 (shared prefix), 3
    and 9, two KV heads, edge and random tokens."""
    b = W.generate(dataclasses.replace(W.config_spec(2), kv_dtype=kv), DEV)
    G = 4
    _sampled(b, [0, 3, 9], [0, 5], token_pick=lambda q: _edge_tokens(q, G), what=f"c3 {kv}")


def test_mixed_step_full_size():
    b = W.generate(W.config_spec(3), DEV)
    G = 8
    # decodes 0, 57, 119 and prefill chunks 120 (2048 tokens) and 127 (392)
    _sampled(b, [0, 57, 119, 120, 127], [0, 7],
             token_pick=lambda q: _edge_tokens(q, G), what="c4")


def test_fp8_long_decode_full_size():
    b = W.generate(W.config_spec(4), DEV)
    L = b.seq_lens
    _sampled(b, [int(L.argmin())], [0, 5], what="c5")


def test_nvfp4_long_decode_full_size():
    """The long-context decode with NVFP4 KV as bench.py times it: the
    shortest and the longest request, two KV heads each."""
    full = W.config_spec(4)
    b = W.generate(dataclasses.replace(full, kv_dtype="nvfp4"), DEV)
    L = b.seq_lens
    _sampled(b, [int(L.argmin()), int(L.argmax())], [0, 5], what="c5 nvfp4")


# ---- invariances -------------------------------------------------------------------

@pytest.mark.parametrize("kv", ["bf16", "nvfp4"])
def test_block_permutation_is_bitwise_invariant(kv):
    s = spec("perm", 32, 8, 16, [1, 70, 1], [3000, 500, 77], kv=kv)
    b = W.generate(s, DEV)
    out1, lse1 = U.gpu_step(b, append=True)
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(5))
    kc = torch.empty_like(b.k_cache)
    vc = torch.empty_like(b.v_cache)
    pd = perm.to(DEV)
    kc[pd] = b.k_cache
    vc[pd] = b.v_cache
    b.k_cache, b.v_cache = kc, vc
    if b.k_scale is not None:
        ks, vs = torch.empty_like(b.k_scale), torch.empty_like(b.v_scale)
        ks[pd] = b.k_scale
        vs[pd] = b.v_scale
        b.k_scale, b.v_scale = ks, vs
    b.block_tables = perm.numpy()[b.block_tables].astype(np.int32)
    out2, lse2 = U.gpu_step(b, append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_run_to_run_deterministic():
    s = spec("det", 64, 8, 16, [1] * 20 + [300], [20000 + 37 * i for i in range(20)] + [4000])
    b = W.generate(s, DEV)
    out1, lse1 = U.gpu_step(b)
    out2, lse2 = U.gpu_step(b, append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_split_prefill_is_deterministic():
    """Key ranges of split prefill items merge in a fixed order: two runs of
    the same step give the same bits."""
    s = spec("det_split", 32, 8, 16, [16, 40], [8208, 3000])
    b = W.generate(s, DEV)
    out1, lse1 = U.gpu_step(b)
    out2, lse2 = U.gpu_step(b, append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_chunked_prefill_matches_one_shot():
    """The same 200 new tokens as one chunk or as chunks of 70/1/129, each
    appended first and attending to history + earlier chunks."""
    s = spec("oneshot", 32, 8, 16, [200], [2200])
    b = W.generate(s, DEV)
    full, full_lse = U.gpu_step(b)
    h = U.make_handle(b)
    m = U.device_meta(b)
    outs, lses, done = [], [], 0
    for c in (70, 1, 129):
        tok = slice(done, done + c)
        qsl = np.array([0, c], np.int32)
        lens = np.array([2000 + done + c], np.int32)
        o = torch.empty_like(b.q[tok])
        l = torch.empty((c, 32), dtype=torch.float32, device=DEV)
        h.attention_varlen(b.q[tok].contiguous(), b.k_cache, b.v_cache,
                           torch.from_numpy(qsl).to(DEV), torch.from_numpy(lens).to(DEV),
                           m["bt"], qsl, lens, out=o, lse=l)
        outs.append(o)
        lses.append(l)
        done += c
    torch.cuda.synchronize()
    chunked = torch.cat(outs).double().cpu().numpy().reshape(-1, 128)
    ref = full.double().cpu().numpy().reshape(-1, 128)
    assert np.abs(chunked - ref).max() <= 1e-2
    np.testing.assert_allclose(torch.cat(lses).cpu().numpy(), full_lse.cpu().numpy(),
                               rtol=0, atol=1e-4)


def test_zeros_fail_the_checks():
    """Negative control: an all-zero output must not pass the parity checks
    at long context, even though it is within the absolute bounds."""
    b = W.generate(W.custom_spec("neg", 64, 8, 64, [1], [300000], kv_dtype="bf16"), DEV)
    sub = W.subset(b, [0], [0])
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    zeros = np.zeros_like(ref)
    assert np.abs(ref).max() < 2e-2          # zeros are within max-abs ...
    with pytest.raises(AssertionError):
        U.check(zeros, ref, ref_lse, ref_lse)   # ... but fail the relative check
    with pytest.raises(AssertionError):
        U.check(ref, ref, ref_lse + 0.01, ref_lse)


# ---- validate mode and API errors on the device ----------------------------------------

@pytest.mark.parametrize("kv", ["bf16", "nvfp4"])
def test_validate_mode_reports_bad_block_ids(kv):
    s = spec("badblk", 8, 2, 16, [1, 5], [40, 60], kv=kv)
    b = W.generate(s, DEV)
    b.block_tables[0, 1] = b.num_blocks + 5      # outside the pool
    h = U.make_handle(b)
    with pytest.raises(pkv.PkvError) as e:
        U.gpu_step(b, handle=h)
    assert e.value.status == 5 and "block-table" in str(e.value)
    h.close()


def test_validate_mode_reports_bad_slots_and_mirror_mismatch():
    s = spec("badslot", 8, 2, 16, [2], [40])
    b = W.generate(s, DEV)
    h = U.make_handle(b)
    m = U.device_meta(b)
    bad = m["slots"].clone()
    bad[0] = b.num_blocks * 16 + 3
    h.write_slots(b.k_new, b.v_new, bad, b.k_cache, b.v_cache)
    with pytest.raises(pkv.PkvError) as e:
        h.check_device_errors()
    assert e.value.status == 5 and "slot" in str(e.value)
    wrong = b.seq_lens.copy()
    m["lens"][0] += 1                            # device copy disagrees
    h.attention_varlen(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"],
                       b.qsl, wrong)
    with pytest.raises(pkv.PkvError) as e:
        h.check_device_errors()
    assert e.value.status == 5 and "mirror" in str(e.value)
    h.check_device_errors()                      # the word was cleared
    h.close()


def test_host_argument_errors():
    s = spec("args", 8, 2, 16, [2], [40])
    b = W.generate(s, DEV)
    h = U.make_handle(b)
    m = U.device_meta(b)
    with pytest.raises(pkv.PkvError) as e:       # stride too small for L
        h.attention_varlen(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"],
                           m["bt"][:, :2].contiguous(), b.qsl, b.seq_lens)
    assert e.value.status == 1
    with pytest.raises(pkv.PkvError) as e:       # more tokens than the handle serves
        h.write_slots(torch.zeros(9, 2, 128, dtype=torch.bfloat16, device=DEV),
                      torch.zeros(9, 2, 128, dtype=torch.bfloat16, device=DEV),
                      torch.zeros(9, dtype=torch.int64, device=DEV), b.k_cache, b.v_cache)
    assert e.value.status == 1
    # empty step: nothing to do, nothing launched
    h.attention_varlen(b.q[:0], b.k_cache, b.v_cache, m["qsl"][:1], m["lens"][:0],
                       m["bt"], np.zeros(1, np.int32), np.zeros(0, np.int32))
    h.close()


