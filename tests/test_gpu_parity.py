"""CUDA path against the fp64 oracle, through the C ABI (GPU only).

Small cases compare every output row.  The five workloads run at full size,
in the launch configuration bench.py times: every output row of the decode
batch and of the long-context E4M3 decode, and every request of the
post-tool-call prefill and of the mixed step on at least 64 rows (the first
and last query tokens, both sides of the Q-tile boundaries, random ones).
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
    ("fp8_prefill_bs128", 16, 4, 128, [200, 2], [1300, 300], "fp8"),
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
    ("split_fp8_bs256", 8, 2, 256, [33, 2], [3000, 700], "fp8"),
    ("split_nvfp4", 32, 8, 16, [40, 1], [6000, 3000], "nvfp4"),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: c[0])
@pytest.mark.parametrize("q_scale", [1.0, 8.0], ids=["normal", "peaked"])
def test_small_cases_every_row(case, q_scale):
    """Quantised pools stage K/V as bf16 for their tensor-core prefill rows
    (the handle has room for the whole step)."""
    name, hq, hkv, bs, ql, sl, kv = case
    b = W.generate(spec(name, hq, hkv, bs, ql, sl, kv=kv), DEV, q_scale=q_scale)
    U.full_parity(b, what=name, peaked=q_scale > 1.0)


# quantised pools whose prefill rows run on the tensor cores
FUSED = [c for c in SWEEP if c[6] != "bf16" and any(q * (c[1] // c[2]) > 8 for q in c[4])
         and c[1] // c[2] <= 128]


@pytest.mark.parametrize("case", FUSED, ids=lambda c: c[0])
@pytest.mark.parametrize("q_scale", [1.0, 8.0], ids=["normal", "peaked"])
def test_small_cases_unstaged_prefill(case, q_scale):
    """The same cases with no staging pools: the prefill kernel converts the
    E4M3 / NVFP4 codes itself (also the path of steps larger than the
    staging pools)."""
    name, hq, hkv, bs, ql, sl, kv = case
    b = W.generate(spec(name, hq, hkv, bs, ql, sl, kv=kv), DEV, q_scale=q_scale)
    U.full_parity(b, what=f"{name} unstaged", peaked=q_scale > 1.0, stage=False)


@pytest.mark.parametrize("kv", ["fp8", "nvfp4"])
def test_staging_is_used_when_it_fits(kv):
    """A step whose prefill contexts fit the staging pools runs the staging
    kernel and then the prefill; one that does not fit runs the prefill
    alone (converting inside), both matching the oracle."""
    s = spec(f"stage_fit_{kv}", 32, 8, 16, [40, 1, 70], [3000, 500, 900], kv=kv)
    b = W.generate(s, DEV)
    sub = W.subset(b, [0, 1, 2])
    ref, ref_lse = U.oracle_subset(sub, s)
    need = W.cdiv(3000, 16) * 16 + W.cdiv(900, 16) * 16     # the two prefill requests
    for cap, staged in ((need, True), (need - 16, False)):
        cfg = pkv.make_config(32, 8, 16, b.num_blocks, 3, s.num_tokens,
                              kv_dtype=U.KV_DTYPES[kv], flags=pkv.FLAG_VALIDATE | pkv.FLAG_TIMING,
                              stage_tokens=cap)
        h = pkv.Handle(cfg)
        b2 = W.generate(s, DEV)
        out, lse = U.gpu_step(b2, handle=h)
        assert h.timing_read(pkv.KERNEL_STAGE)[0] == (1 if staged else 0)
        assert h.timing_read(pkv.KERNEL_PREFILL)[0] == 1
        h.close()
        got, got_lse = U.gpu_rows(out, lse, sub)
        U.check(got, ref, got_lse, ref_lse, kv, f"stage_fit {kv} cap {cap}", scaled=True)


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
    U.check(got, ref, got_lse, ref_lse, kv, f"mixed_modes {kv}", scaled=True)
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


# ---- the five workloads at full size ------------------------------------------------
#
# The step runs once on the GPU as bench.py launches it; its outputs are kept
# on the host and the batch is dropped.  The pools are then drawn again from
# the same seeds (the generator is deterministic), so the oracle reads the
# generator's contents and does its own append: none of its inputs passes
# through the CUDA path.  The oracle evaluates the chosen rows group by group
# (a few requests at a time, bounded host memory).

def _workload_outputs(spec):
    b = W.generate(spec, DEV)
    out, lse = U.gpu_step(b)
    res = out.cpu(), lse.cpu()
    del b, out, lse
    torch.cuda.empty_cache()
    return res


def _edge_tokens(q, G, seed, n_random=4):
    """Query tokens to check in a request of q new tokens: the first and last
    ones, both sides of every Q-tile boundary of the first and last prefill
    items (tiles of G * floor(128 / G) rows, two per item) and n_random more."""
    per_tile = max(1, 128 // G)
    picks = {0, 1, q - 2, q - 1}
    for k in (1, 2, 3):
        for c in (k * per_tile, q - k * per_tile):
            picks |= {c - 1, c}
    rng = np.random.default_rng(seed)
    picks |= set(rng.integers(0, q, n_random).tolist())
    return sorted(p for p in picks if 0 <= p < q)


def _rows(sub, G, token_pick=None, all_heads=True):
    """Row indices (token * Hq_sub + head) of a subset: the tokens
    token_pick(q, request) of each request (all with None), with all query
    heads, or one query head per KV head (the head within the group rotates
    with the token)."""
    hq = len(sub["heads"])
    rows = []
    for r in range(len(sub["qsl"]) - 1):
        a = int(sub["qsl"][r])
        q = int(sub["qsl"][r + 1]) - a
        toks = range(q) if token_pick is None else token_pick(q, r)
        for t in toks:
            if all_heads:
                rows.extend((a + t) * hq + h for h in range(hq))
            else:
                rows.extend((a + t) * hq + kvh * G + (t + kvh) % G for kvh in range(hq // G))
    return np.asarray(rows, np.int64)


def _check_groups(spec, outputs, groups, token_pick=None, all_heads=True, what=""):
    """Regenerate the pools and compare the rows of each group of requests
    with the oracle; returns the worst figures over all groups."""
    out, lse = outputs
    b = W.generate(spec, DEV)
    G = spec.hq // spec.hkv
    worst = dict(max_abs=0.0, mean_abs=0.0, rel=0.0, lse=0.0, rows=0)
    for grp in groups:
        sub = W.subset(b, list(grp))
        pick = None if token_pick is None else (lambda q, r: token_pick(q, grp[r]))
        rows = _rows(sub, G, pick, all_heads)
        ref, ref_lse = U.oracle_subset(sub, spec, rows=rows)
        got, got_lse = U.gpu_rows(out, lse, sub, rows)
        st = U.check(got, ref, got_lse, ref_lse, spec.kv_dtype, f"{what} requests {grp}")
        for k in ("max_abs", "mean_abs", "rel", "lse"):
            worst[k] = max(worst[k], st[k])
        worst["rows"] += len(rows)
    del b
    torch.cuda.empty_cache()
    print(f"{what}: {worst}")
    return worst


def _chunks(ids, n):
    ids = list(ids)
    return [ids[i:i + n] for i in range(0, len(ids), n)]


def test_decode_batch_full_size():
    """Decode batch: every output row (64 requests x 32 heads)."""
    spec = W.config_spec(1)
    res = _workload_outputs(spec)
    _check_groups(spec, res, _chunks(range(spec.num_seqs), 16), what="c2")


@pytest.mark.parametrize("kv", ["bf16", "fp8", "nvfp4"])
def test_post_tool_prefill_full_size(kv):
    """The post-tool-call prefill as bench.py times it (bf16, and the E4M3 /
    NVFP4 KV variants of its secondary lines): all 16 sessions, each on the
    first, last, tile-boundary and random query tokens; every query head
    with bf16 KV, one query head per KV head (rotating within the group)
    with quantised KV."""
    spec = dataclasses.replace(W.config_spec(2), kv_dtype=kv)
    res = _workload_outputs(spec)
    G = spec.hq // spec.hkv
    _check_groups(spec, res, _chunks(range(spec.num_seqs), 4),
                  token_pick=lambda q, i: _edge_tokens(q, G, 100 + i),
                  all_heads=kv == "bf16", what=f"c3 {kv}")


def test_mixed_step_full_size():
    """Mixed step: every row of the 120 decodes (64 heads each) and, for each
    of the 8 prefill chunks, the first, last, tile-boundary and random
    tokens on one query head per KV head (>= 128 rows per chunk)."""
    spec = W.config_spec(3)
    res = _workload_outputs(spec)
    G = spec.hq // spec.hkv
    _check_groups(spec, res, _chunks(range(120), 20), what="c4 decodes")
    _check_groups(spec, res, _chunks(range(120, 128), 2),
                  token_pick=lambda q, i: _edge_tokens(q, G, 200 + i),
                  all_heads=False, what="c4 chunks")


def test_fp8_long_decode_full_size():
    """Long-context decode with E4M3 KV: every output row (8 requests of
    512K-1M keys x 64 heads), the longest request included."""
    spec = W.config_spec(4)
    res = _workload_outputs(spec)
    _check_groups(spec, res, _chunks(range(spec.num_seqs), 2), what="c5")


def test_nvfp4_long_decode_full_size():
    """The long-context decode with NVFP4 KV as bench.py times it: every row
    of the shortest and the longest request, and one query head per KV head
    of the other six."""
    spec = dataclasses.replace(W.config_spec(4), kv_dtype="nvfp4")
    res = _workload_outputs(spec)
    L = np.asarray(spec.seq_lens)
    ends = sorted({int(L.argmin()), int(L.argmax())})
    rest = [i for i in range(spec.num_seqs) if i not in ends]
    _check_groups(spec, res, [[i] for i in ends], what="c5 nvfp4 shortest/longest")
    _check_groups(spec, res, _chunks(rest, 3), token_pick=lambda q, i: [0],
                  all_heads=False, what="c5 nvfp4 others")


# ---- quantised KV at realistic magnitudes ------------------------------------------------
#
# KV entries of real models are far from N(0, 1): with K and V drawn with
# standard deviation sigma, E4M3 block scales are about 1e-2 sigma (1e-3 to
# 1e-5 here) and NVFP4 block scales about 1.5e-3 sigma.  The queries are
# drawn with 1/sigma so that the scores keep their N(0, 1) spread.  Decode
# (64K and 100K keys) and tensor-core prefill rows (40 tokens over 70K keys),
# every row, with the relative-L2 and log-sum-exp checks.

@pytest.mark.parametrize("kv", ["fp8", "nvfp4"])
@pytest.mark.parametrize("sigma", [1e-1, 1e-2, 1e-3])
def test_quantised_kv_at_small_magnitudes(kv, sigma):
    s = spec(f"mag_{kv}_{sigma:g}", 8, 2, 64, [1, 1, 40, 1], [65536, 100000, 70040, 3000],
             kv=kv)
    b = W.generate(s, DEV, q_scale=1.0 / sigma, kv_sigma=sigma)
    st = U.full_parity(b, what=f"{kv} sigma {sigma:g}")
    print(f"{kv} sigma {sigma:g}: {st}")


def test_fp8_value_scales_that_jump_between_blocks():
    """E4M3 pools whose V block scales differ by factors of 2^-16 .. 1 from
    block to block (and K scales by 2^-2 .. 2^2): decode and prefill rows,
    every row."""
    s = spec("jump_fp8", 8, 2, 16, [1, 1, 30, 1], [20000, 7000, 9000, 33], kv="fp8")
    b = W.generate(s, DEV, q_scale=0.5)
    g = torch.Generator(device="cpu").manual_seed(77)
    ev = torch.randint(-16, 1, b.v_scale.shape, generator=g).to(DEV)
    ek = torch.randint(-2, 3, b.k_scale.shape, generator=g).to(DEV)
    b.v_scale.mul_(torch.pow(2.0, ev.float()))
    b.k_scale.mul_(torch.pow(2.0, ek.float()))
    st = U.full_parity(b, what="jump_fp8", peaked=True)
    print(f"jump_fp8: {st}")


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


def test_single_long_request_many_ranges():
    """One 600K-token decode split over the whole machine (over 100 key
    ranges per (request, KV head) pair, merged by the wide merge kernel):
    every row against the oracle, and the same bits on a second run."""
    s = spec("long_one", 32, 8, 16, [1], [600_000])
    b = W.generate(s, DEV)
    sub = W.subset(b, [0])
    out1, lse1 = U.gpu_step(b)
    out2, lse2 = U.gpu_step(b, append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    got, got_lse = U.gpu_rows(out1, lse1, sub)
    st = U.check(got, ref, got_lse, ref_lse, "bf16", "long_one")
    print(f"long_one: {st}")


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


@pytest.mark.parametrize("kv", ["fp8", "nvfp4"])
def test_validate_mode_reports_scales_above_the_cap(kv):
    """E4M3 and NVFP4 block scales must be at most 16; validate mode checks
    every block in use before the attention kernels and reports
    PKV_ERR_DEVICE_CHECK."""
    s = spec("bigscale", 8, 2, 16, [1, 5], [40, 60], kv=kv)
    b = W.generate(s, DEV)
    h = U.make_handle(b)
    m = U.device_meta(b)
    h.write_slots(b.k_new, b.v_new, m["slots"], b.k_cache, b.v_cache, b.k_scale, b.v_scale)
    h.check_device_errors()
    b.v_scale[int(b.block_tables[1, 2]), 1] = 20.0
    h.attention_varlen(b.q, b.k_cache, b.v_cache, m["qsl"], m["lens"], m["bt"], b.qsl,
                       b.seq_lens, k_scale=b.k_scale, v_scale=b.v_scale)
    with pytest.raises(pkv.PkvError) as e:
        h.check_device_errors()
    assert e.value.status == 5 and "scale" in str(e.value)
    h.close()


def test_a_device_wait_that_runs_out_is_reported():
    """Failure detection without a fault: pkv_wait_selftest waits, through
    the kernels' bounded-wait helper, on a barrier nothing arrives at; the
    wait gives up after 10 us, the timeout comes back from
    pkv_check_device_errors as PKV_ERR_TIMEOUT, the word is cleared, and the
    handle still computes a correct step."""
    s = spec("timeout", 8, 2, 16, [1, 20], [300, 700])
    b = W.generate(s, DEV)
    h = U.make_handle(b)
    h.check_device_errors()
    h.wait_selftest(10_000)
    with pytest.raises(pkv.PkvError) as e:
        h.check_device_errors()
    assert e.value.status == 6
    h.check_device_errors()                      # cleared
    with pytest.raises(pkv.PkvError) as e:       # the limit is checked on the host
        h.wait_selftest(0)
    assert e.value.status == 1
    sub = W.subset(b, [0, 1])
    out, lse = U.gpu_step(b, handle=h)
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    got, got_lse = U.gpu_rows(out, lse, sub)
    U.check(got, ref, got_lse, ref_lse, "bf16", "after timeout", scaled=True)
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


