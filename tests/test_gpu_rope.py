"""Rotary embedding fused with the KV append (pkv_rope_write_slots) against
the oracle's fp64 RoPE and its own append, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _table(max_pos, d=128, base=10000.0):
    inv = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).double().numpy()


def _bf16_ulp_ok(got_bits, ref_f64, ref_bits, x_bits, neox):
    """Equal bits, or the neighbouring bf16 value where the exact result lies
    within the fp32 arithmetic's error of the rounding midpoint: the GPU
    rounds x_b sin and then the fused multiply-add in fp32, so its error is
    at most 2^-24 (|x_b sin| + |y|) <= 2^-23 (|x_a| + |x_b|)."""
    same = got_bits == ref_bits
    g, r = _f(got_bits), _f(ref_bits)
    x = np.abs(_f(x_bits))
    d = x.shape[-1]
    partner = np.arange(d) ^ (d // 2 if neox else 1)
    bound = 2.0 ** -23 * (x + x[..., partner])
    near = np.abs(ref_f64 - (g + r) / 2) <= bound
    adjacent = np.abs(got_bits.astype(np.int32) - ref_bits.astype(np.int32)) <= 1
    return bool(np.all(same | (near & adjacent))), float(np.mean(~same))


@pytest.mark.parametrize("kv,neox", [("bf16", True), ("bf16", False), ("fp8", True),
                                     ("nvfp4", False)])
def test_rope_append_matches_the_oracle(kv, neox):
    s = W.custom_spec(f"rope_{kv}", 32, 8, 16 if kv == "bf16" else 64, [37, 1, 200],
                      [100, 5000, 260], seed=31, kv_dtype=kv)
    b = W.generate(s, DEV)
    b.slot_mapping[3] = -1                                  # a padding token
    T = b.q.shape[0]
    rng = np.random.default_rng(7)
    max_pos = 6000
    tab = _table(max_pos)
    pos = rng.integers(0, max_pos, T).astype(np.int64)
    q0 = W.bf16_bits(b.q)
    kc0, vc0 = W.host_pool(b, "k"), W.host_pool(b, "v")
    h = U.make_handle(b)
    h.rope_write_slots(b.q, b.k_new, b.v_new, torch.from_numpy(pos).to(DEV),
                       torch.from_numpy(tab).to(DEV),
                       torch.from_numpy(b.slot_mapping).to(DEV), b.k_cache, b.v_cache,
                       neox=neox, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    h.check_device_errors()
    # q: rotated in place
    qf, qbits = oracle.rope(q0, pos, tab, neox=neox)
    ok, frac = _bf16_ulp_ok(W.bf16_bits(b.q), qf, qbits, q0, neox)
    assert ok and frac < 1e-3, frac
    # K rotated then appended, V appended: the oracle's append of its own
    # rotated K must agree with the pools wherever the rotated bf16 K agree
    kf, kbits = oracle.rope(W.bf16_bits(b.k_new), pos, tab, neox=neox)
    ks = b.k_scale.cpu().numpy() if kv != "bf16" else None
    vs = b.v_scale.cpu().numpy() if kv != "bf16" else None
    oracle.write_slots(kc0, vc0, kbits, W.bf16_bits(b.v_new), b.slot_mapping,
                       k_scale=ks, v_scale=vs)
    assert np.array_equal(W.host_pool(b, "v"), vc0)
    kg = W.host_pool(b, "k")
    diff = kg != kc0
    if kv == "nvfp4":
        # a rotated K element one bf16 ulp off can move its micro block's
        # scale and so all 16 codes; such blocks are rare
        assert diff.mean() < 1e-2
        h.close()
        return
    assert diff.mean() < 1e-3
    if kv == "bf16":
        rows = np.nonzero(diff.any(-1))
        assert len(rows[0]) == 0 or np.all(np.abs(kg.astype(np.int32) - kc0.astype(np.int32))[diff] <= 1)
    else:
        # a differing code is the neighbour of the oracle's (same sign, magnitude +-1)
        a, c = kg[diff].astype(np.int32), kc0[diff].astype(np.int32)
        assert np.all((a & 0x80) == (c & 0x80)) and np.all(np.abs((a & 0x7F) - (c & 0x7F)) <= 1)
    h.close()


def test_out_of_range_position_is_reported_and_skipped():
    s = W.custom_spec("rope_bad", 8, 2, 16, [4], [20], seed=5)
    b = W.generate(s, DEV)
    tab = _table(16)
    pos = torch.tensor([0, 3, 16, 2], dtype=torch.int64, device=DEV)   # 16 is out of range
    q0 = b.q.clone()
    h = U.make_handle(b)
    h.rope_write_slots(b.q, b.k_new, b.v_new, pos, torch.from_numpy(tab).to(DEV),
                       torch.from_numpy(b.slot_mapping).to(DEV), b.k_cache, b.v_cache)
    with pytest.raises(pkv.PkvError) as e:
        h.check_device_errors()
    assert "rotary position" in str(e.value)
    assert torch.equal(b.q[2], q0[2])                   # that token untouched
    assert torch.equal(b.q[0], q0[0])                   # position 0: identity
    h.close()
