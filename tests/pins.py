"""Pins of the fp64 oracle against facts other than itself.

Each ``pin_*`` function takes an oracle library handle and raises
AssertionError when the oracle disagrees with:

* a library routine on the special case it reduces to (torch's fp64
  scaled-dot-product attention on contiguous K/V; torch's E4M3 cast),
* a closed form (single key, uniform scores, needle key, the E4M3 grid),
* an invariance the definition implies (physical block permutation, chunked
  versus one-shot prefill, decode = prefill of one token, GQA = MHA with
  repeated KV heads, the log-sum-exp merge of disjoint key sets).

``tests/test_oracle_pins.py`` runs them on the oracle; and
``tests/test_oracle_mutations.py`` runs them on copies of the oracle with
planted mistakes, each of which must fail at least one pin.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

import oracle

NAN16 = 0x7FC0


def _bf16(rng: np.random.Generator, shape, scale=1.0) -> np.ndarray:
    x = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def _f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Paged:
    """A small paged problem built from contiguous per-sequence K/V.

    The test places each sequence's rows into randomly chosen physical blocks
    (the inverse of the gather under test); everything else is NaN poison and
    table entries past cdiv(L, bs) are INT32_MAX.
    """

    def __init__(self, rng, hq, hkv, d, bs, q_lens, seq_lens, spare=3,
                 q_scale=1.0):
        self.hq, self.hkv, self.d, self.bs = hq, hkv, d, bs
        self.q_lens = list(q_lens)
        self.seq_lens = list(seq_lens)
        B = len(seq_lens)
        nblk = [-(-L // bs) for L in seq_lens]
        self.num_blocks = sum(nblk) + spare
        perm = rng.permutation(self.num_blocks)
        self.bt = np.full((B, max(nblk) + 2), np.iinfo(np.int32).max, np.int32)
        self.kc = np.full((self.num_blocks, hkv, bs, d), NAN16, np.uint16)
        self.vc = np.full_like(self.kc, NAN16)
        self.K = []   # contiguous [L, hkv, d] bits per sequence
        self.V = []
        nxt = 0
        for i, L in enumerate(seq_lens):
            ids = perm[nxt:nxt + nblk[i]]
            nxt += nblk[i]
            self.bt[i, :nblk[i]] = ids
            K = _bf16(rng, (L, hkv, d))
            V = _bf16(rng, (L, hkv, d))
            self.K.append(K)
            self.V.append(V)
            for p in range(L):
                self.kc[ids[p // bs], :, p % bs, :] = K[p]
                self.vc[ids[p // bs], :, p % bs, :] = V[p]
        self.qsl = np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)
        self.T = int(self.qsl[-1])
        self.q = _bf16(rng, (self.T, hq, d), q_scale)
        self.scale = 1.0 / math.sqrt(d)

    def run(self, lib, rows=None, k_range=None, shard=None):
        return oracle.attention(self.kc, self.vc, self.q, self.qsl,
                                np.asarray(self.seq_lens, np.int32), self.bt,
                                self.scale, rows=rows, k_range=k_range, shard=shard,
                                lib=lib)

    def sdpa(self, keep=None):
        """torch fp64 scaled_dot_product_attention on the contiguous K/V,
        with one extra zero key whose value is a unit vector in an extra
        column: its weight w0 = 1 / (1 + sum_j exp(s_j)) gives
        lse = ln(1/w0 - 1).  ``keep(j)`` (optional) further restricts the keys;
        a row that keeps none gets out 0 and lse -inf.  Returns
        (out [T*hq, d], lse [T*hq])."""
        G = self.hq // self.hkv
        outs = np.zeros((self.T, self.hq, self.d))
        lses = np.zeros((self.T, self.hq))
        for i, L in enumerate(self.seq_lens):
            qi = self.q_lens[i]
            a = int(self.qsl[i])
            q = torch.from_numpy(_f64(self.q[a:a + qi])).permute(1, 0, 2)
            k = torch.from_numpy(_f64(self.K[i])).permute(1, 0, 2)
            v = torch.from_numpy(_f64(self.V[i])).permute(1, 0, 2)
            k = k.repeat_interleave(G, dim=0)
            v = v.repeat_interleave(G, dim=0)
            # extra key (score 0) and extra value column
            k = torch.cat([torch.zeros(self.hq, 1, self.d, dtype=k.dtype), k], 1)
            v = torch.cat([v, torch.zeros(self.hq, L, 1, dtype=v.dtype)], 2)
            e0 = torch.zeros(self.hq, 1, self.d + 1, dtype=v.dtype)
            e0[:, :, self.d] = 1.0
            v = torch.cat([e0, v], 1)
            h = L - qi
            pos = torch.arange(qi)[:, None] + h
            j = torch.arange(L)[None, :]
            vis = j <= pos
            if keep is not None:
                vis = vis & torch.tensor([bool(keep(x)) for x in range(L)])[None, :]
            mask = torch.cat([torch.ones(qi, 1, dtype=torch.bool), vis], 1)
            # scale the scores to the original ones; the extra column is
            # exactly sum_j w_j * 0 + w0 * 1
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None], k[None], v[None], attn_mask=mask[None, None],
                scale=self.scale)[0]
            w0 = o[:, :, self.d]
            body = o[:, :, :self.d] / (1.0 - w0)[:, :, None]
            none = ~vis.any(1)                        # rows with no kept key
            body[:, none, :] = 0.0
            outs[a:a + qi] = body.permute(1, 0, 2).numpy()
            lses[a:a + qi] = torch.log(1.0 / w0 - 1.0).permute(1, 0).numpy()
        return outs.reshape(-1, self.d), lses.reshape(-1)


# ---- attention pins ---------------------------------------------------------

TINY_CASES = [
    # hq, hkv, d, bs, q_lens, seq_lens
    (2, 1, 8, 1, [3], [5]),
    (4, 2, 16, 2, [1, 4, 2], [7, 4, 9]),
    (8, 2, 16, 16, [5, 1, 17], [40, 70, 17]),
    (4, 4, 8, 16, [16], [33]),
    (8, 1, 32, 4, [2, 3], [2, 11]),
]


def pin_sdpa(lib):
    """Special case = a library routine: paged attention equals torch fp64
    SDPA (bottom-right causal mask, GQA by repetition) on the same rows."""
    rng = np.random.default_rng(11)
    for hq, hkv, d, bs, ql, sl in TINY_CASES:
        P = Paged(rng, hq, hkv, d, bs, ql, sl)
        out, lse = P.run(lib)
        ref, ref_lse = P.sdpa()
        assert np.all(np.isfinite(out)), "poison leaked"
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-9)
    # one full-width head_dim 128 case
    P = Paged(rng, 8, 2, 128, 16, [6, 1], [37, 20], q_scale=3.0)
    out, lse = P.run(lib)
    ref, ref_lse = P.sdpa()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-9)


def pin_block_permutation(lib):
    """Renaming physical blocks (moving their contents along) leaves every
    output bit unchanged."""
    rng = np.random.default_rng(12)
    P = Paged(rng, 8, 2, 16, 4, [3, 1, 6], [21, 9, 30], spare=5)
    out, lse = P.run(lib)
    perm = rng.permutation(P.num_blocks)
    kc = np.empty_like(P.kc)
    vc = np.empty_like(P.vc)
    kc[perm] = P.kc
    vc[perm] = P.vc
    bt = P.bt.copy()
    for i, L in enumerate(P.seq_lens):
        n = -(-L // P.bs)
        bt[i, :n] = perm[P.bt[i, :n]]
    out2, lse2 = oracle.attention(kc, vc, P.q, P.qsl,
                                  np.asarray(P.seq_lens, np.int32), bt, P.scale,
                                  lib=lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_chunked_prefill(lib):
    """One-shot prefill of l_incr tokens equals the same tokens run as
    chunks, each appended with write_slots and attending to the history plus
    the earlier chunks (bitwise); decode = the last row of a prefill."""
    rng = np.random.default_rng(13)
    hq, hkv, d, bs = 4, 2, 16, 4
    hist, incr = 13, 11
    L = hist + incr
    P = Paged(rng, hq, hkv, d, bs, [incr], [L])
    full, full_lse = P.run(lib)
    # pool holding only the history; new rows arrive by write_slots
    kc = P.kc.copy()
    vc = P.vc.copy()
    bt = P.bt
    for p in range(hist, L):
        kc[bt[0, p // bs], :, p % bs, :] = NAN16
        vc[bt[0, p // bs], :, p % bs, :] = NAN16
    done = hist
    outs, lses = [], []
    for c in (4, 1, 6):
        new = np.arange(done, done + c)
        slots = (bt[0, new // bs].astype(np.int64) * bs + new % bs)
        oracle.write_slots(kc, vc, P.K[0][new], P.V[0][new], slots, lib=lib)
        q = P.q[new - hist]
        o, l = oracle.attention(kc, vc, q, np.array([0, c], np.int32),
                                np.array([done + c], np.int32), bt, P.scale,
                                lib=lib)
        outs.append(o)
        lses.append(l)
        done += c
    assert np.array_equal(np.concatenate(outs), full)
    assert np.array_equal(np.concatenate(lses), full_lse)
    # decode of the last token over the full context
    o, l = oracle.attention(kc, vc, P.q[-1:], np.array([0, 1], np.int32),
                            np.array([L], np.int32), bt, P.scale, lib=lib)
    assert np.array_equal(o, full[-hq:]) and np.array_equal(l, full_lse[-hq:])


def pin_closed_forms(lib):
    """L = 1: out = V_0 and lse = s_0.  Q = 0: out = mean(V_0..V_pos) and
    lse = ln(pos + 1).  A needle key scoring 40 above the rest: out = its V."""
    rng = np.random.default_rng(14)
    d = 16
    P = Paged(rng, 2, 1, d, 16, [1], [1])
    out, lse = P.run(lib)
    v0 = _f64(P.V[0][0, 0])
    s0 = P.scale * (_f64(P.q[0]) @ _f64(P.K[0][0, 0]))    # one score per head
    assert np.array_equal(out[0], v0) and np.array_equal(out[1], v0)
    np.testing.assert_allclose(lse, s0, rtol=0, atol=1e-13)

    P = Paged(rng, 4, 2, d, 4, [5], [19])
    P.q[:] = 0
    out, lse = P.run(lib)
    hist = 19 - 5
    for t in range(5):
        pos = hist + t
        for h in range(4):
            ref = _f64(P.V[0][:pos + 1, h // 2]).mean(axis=0)
            np.testing.assert_allclose(out[t * 4 + h], ref, rtol=0, atol=1e-14)
            assert abs(lse[t * 4 + h] - math.log(pos + 1)) < 1e-13

    P = Paged(rng, 1, 1, d, 4, [1], [23])
    P.q[:] = 0
    one = np.uint16(0x3F80)      # bf16 1.0
    P.q[0, 0, 0] = one
    needle = 9
    for p in range(23):
        row = P.K[0][p, 0].copy()
        row[0] = 0
        if p == needle:
            row[0] = np.uint16(0x4220)   # bf16 40.0
        blk = P.bt[0, p // 4]
        P.kc[blk, 0, p % 4] = row
    P.scale = 1.0
    out, lse = P.run(lib)
    np.testing.assert_allclose(out[0], _f64(P.V[0][needle, 0]), rtol=0,
                               atol=1e-14)
    assert abs(lse[0] - (40 + math.log1p(22 * math.exp(-40)))) < 1e-12


def pin_gqa_is_repeated_mha(lib):
    """GQA with group G equals MHA (G = 1) over KV heads repeated G times."""
    rng = np.random.default_rng(15)
    G = 4
    P = Paged(rng, 8, 2, 16, 4, [3, 1], [10, 6])
    out, lse = P.run(lib)
    kc = np.repeat(P.kc, G, axis=1)
    vc = np.repeat(P.vc, G, axis=1)
    out2, lse2 = oracle.attention(kc, vc, P.q, P.qsl,
                                  np.asarray(P.seq_lens, np.int32), P.bt,
                                  P.scale, lib=lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_lse_merge(lib):
    """Partial results over any partition of the keys merge, through their
    log-sum-exp, into the unsplit result; a part with no key is neutral."""
    rng = np.random.default_rng(16)
    P = Paged(rng, 4, 2, 16, 4, [2], [45], q_scale=2.0)
    full, full_lse = P.run(lib)
    cuts = [0, 7, 8, 30, 44, 46]
    parts = [P.run(lib, k_range=(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
    parts.append(P.run(lib, k_range=(100, 200)))   # empty: lse = -inf
    for r in range(full.shape[0]):
        lses = np.array([p[1][r] for p in parts])
        os_ = np.stack([p[0][r] for p in parts])
        o, l = oracle.lse_merge(lses, os_, lib=lib)
        np.testing.assert_allclose(o, full[r], rtol=0, atol=1e-13)
        assert abs(l - full_lse[r]) < 1e-12
        # order does not matter
        o2, l2 = oracle.lse_merge(lses[::-1].copy(), os_[::-1].copy(), lib=lib)
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-15)


def pin_context_parallel_shards(lib):
    """Decode context parallelism (page "vLLM Agentic 推理｜面向 Agent 负载的推理优化",
    sections 4.3.1 and 4.3.3): with interleave 1, token i belongs to rank
    i % N; with runs of k tokens, run i // k belongs to rank (i // k) % N.
    Each rank's partial equals torch fp64 SDPA over exactly its keys, a
    rank with no visible key gives (0, -inf), and the log-sum-exp merge of
    all ranks' partials is the unsharded result."""
    rng = np.random.default_rng(19)
    P = Paged(rng, 8, 2, 16, 4, [1, 3, 1, 1], [29, 41, 3, 1], q_scale=2.0)
    full, full_lse = P.run(lib)
    for n, k in ((2, 1), (3, 1), (8, 1), (2, 4), (3, 5), (2, 16)):
        parts = []
        for r in range(n):
            if k == 1:
                keep = (lambda r: lambda i: i % n == r)(r)          # token i -> rank i % N
            else:
                keep = (lambda r: lambda i: (i // k) % n == r)(r)   # run i // k -> rank
            out, lse = P.run(lib, shard=(n, r, k))
            ref, ref_lse = P.sdpa(keep=keep)
            assert np.all(np.isfinite(out)), "poison leaked"
            np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
            fin = np.isfinite(ref_lse)
            assert np.array_equal(np.isfinite(lse), fin), (n, k, r)
            np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-9)
            parts.append((out, lse))
        for row in range(full.shape[0]):
            o, l = oracle.lse_merge(np.array([p[1][row] for p in parts]),
                                    np.stack([p[0][row] for p in parts]), lib=lib)
            np.testing.assert_allclose(o, full[row], rtol=0, atol=1e-12)
            assert abs(l - full_lse[row]) < 1e-11


# ---- rotary embedding pins ---------------------------------------------------------

def _rope_table(rng, max_pos, d=128):
    ang = rng.uniform(-math.pi, math.pi, (max_pos, d // 2))
    ang[0] = 0.0                                        # position 0: identity
    return np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)


def pin_rope_is_a_complex_rotation(lib):
    """Library routine: each pair (a, b) rotates like the complex number
    x_a + i x_b multiplied by cos + i sin (torch complex128), for both pair
    layouts; position 0 with angle 0 is the identity (bit-exact)."""
    rng = np.random.default_rng(23)
    x = _bf16(rng, (7, 3, 128), 3.0)
    tab = _rope_table(rng, 50)
    pos = np.array([0, 1, 49, 7, 7, 0, 30], np.int64)
    xf = torch.from_numpy(_f64(x))
    c = torch.from_numpy(tab[pos, :64].astype(np.float64))[:, None, :]
    sn = torch.from_numpy(tab[pos, 64:].astype(np.float64))[:, None, :]
    rot = torch.complex(c, sn)
    for neox in (True, False):
        y, bits = oracle.rope(x, pos, tab, neox=neox, lib=lib)
        if neox:
            z = torch.complex(xf[..., :64], xf[..., 64:]) * rot
            ref = torch.cat([z.real, z.imag], -1)
        else:
            z = torch.view_as_complex(xf.reshape(7, 3, 64, 2).contiguous()) * rot
            ref = torch.view_as_real(z).reshape(7, 3, 128)
        np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-14)
        assert np.array_equal(bits[pos == 0], x[pos == 0])


def pin_bf16_round(lib):
    """Rounding to bf16 equals torch's float32 -> bfloat16 cast (nearest,
    ties to even) on float32 values: random, ties, subnormals, overflow."""
    rng = np.random.default_rng(29)
    v = (rng.standard_normal(4000) * np.exp(rng.uniform(-85, 85, 4000))).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7),
                     2.0 ** -130, 3.5 * 2.0 ** -133, 2.0 ** -134, 3.4e38, -3.39e38,
                     0.0, -0.0], np.float32)
    v = np.concatenate([v, ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(a), lib=lib) for a in v], np.uint16)
    assert np.array_equal(got, ref), v[got != ref][:5]


# ---- KV append and FP8 pins -----------------------------------------------------

def pin_write_slots_bf16(lib):
    """Appended rows land bit-exactly at their slots; skipped (-1) tokens
    and every other byte of the pool keep their poison."""
    rng = np.random.default_rng(17)
    nb, hkv, bs, d = 9, 2, 4, 8
    kc = np.full((nb, hkv, bs, d), NAN16, np.uint16)
    vc = kc.copy()
    T = 10
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    kn = _bf16(rng, (T, hkv, d))
    vn = _bf16(rng, (T, hkv, d))
    oracle.write_slots(kc, vc, kn, vn, slots, lib=lib)
    touched = np.zeros((nb, bs), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc[s // bs, :, s % bs], kn[t])
        assert np.array_equal(vc[s // bs, :, s % bs], vn[t])
        touched[s // bs, s % bs] = True
    untouched = ~touched[:, None, :].repeat(hkv, axis=1)
    assert np.all(kc[untouched] == NAN16) and np.all(vc[untouched] == NAN16)


def pin_e4m3_decode(lib):
    """All 256 codes decode as torch's float8_e4m3fn does; grid landmarks
    from the format definition."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([lib.pko_e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2
    assert np.array_equal(ref[~nan], got[~nan])
    assert lib.pko_e4m3_value(0x7E) == 448.0
    assert lib.pko_e4m3_value(0x01) == 2.0 ** -9
    assert lib.pko_e4m3_value(0x08) == 2.0 ** -6
    assert lib.pko_e4m3_value(0x38) == 1.0
    assert lib.pko_e4m3_value(0xB8) == -1.0


def pin_e4m3_encode(lib):
    """Encoding rounds to nearest with ties to even (as torch's cast does on
    in-range values) and saturates at +-448."""
    enc = lib.pko_e4m3_encode
    for c in range(256):
        v = lib.pko_e4m3_value(c)
        if not math.isnan(v):
            assert enc(v) == c or (v == 0 and enc(v) in (0, 0x80))
    rng = np.random.default_rng(18)
    x = np.concatenate([rng.standard_normal(20000) * 50,
                        rng.standard_normal(5000) * 0.01,
                        rng.uniform(-447.9, 447.9, 5000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([enc(float(v)) for v in x], dtype=np.uint8)
    inr = np.abs(x) < 448
    assert np.array_equal(ref[inr], got[inr])
    # ties: 1.0625 lies halfway between 1.0 (even) and 1.125 -> 1.0;
    # 1.1875 halfway between 1.125 and 1.25 (even) -> 1.25;
    # 2^-10 halfway between 0 and 2^-9 -> 0; 3*2^-10 -> 2^-8 (even)
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A
    assert enc(2.0 ** -10) == 0x00 and enc(3 * 2.0 ** -10) == 0x02
    for big in (448.0, 460.0, 464.0, 479.0, 1e6, float("inf")):
        assert enc(big) == 0x7E and enc(-big) == 0xFE
    assert enc(float("nan")) & 0x7F == 0x7F


def pin_write_slots_fp8(lib):
    """FP8 append: code = E4M3(x / scale) with the quotient in fp32; checked
    against torch's fp32 division and E4M3 cast for in-range quotients."""
    rng = np.random.default_rng(19)
    nb, hkv, bs, d = 5, 2, 4, 16
    kc = np.full((nb, hkv, bs, d), 0x7F, np.uint8)
    vc = kc.copy()
    ks = rng.uniform(0.005, 0.02, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.005, 0.02, (nb, hkv)).astype(np.float32)
    T = 6
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    kn = _bf16(rng, (T, hkv, d))
    vn = _bf16(rng, (T, hkv, d))
    oracle.write_slots(kc, vc, kn, vn, slots, k_scale=ks, v_scale=vs, lib=lib)
    for t, s in enumerate(slots):
        b, o = s // bs, s % bs
        for src, cache, sc in ((kn, kc, ks), (vn, vc, vs)):
            x = torch.from_numpy(_f64(src[t]).astype(np.float32))
            qt = x / torch.from_numpy(sc[b])[:, None]
            sat = qt.abs() >= 448
            ref = qt.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(cache[b, :, o][~sat.numpy()], ref[~sat.numpy()])
            assert np.all((cache[b, :, o][sat.numpy()] & 0x7F) == 0x7E)


def pin_fp8_attention(lib):
    """FP8 pools attend over the exact dequantised values e4m3(code)*scale:
    same result as a bf16-free fp64 evaluation through SDPA."""
    rng = np.random.default_rng(20)
    hq, hkv, d, bs = 4, 2, 16, 8
    L, ql = 21, 3
    nb = 5
    codes_k = rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8)
    codes_v = rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8)
    codes_k[(codes_k & 0x7F) == 0x7F] = 0x10   # no NaN codes in used rows
    codes_v[(codes_v & 0x7F) == 0x7F] = 0x10
    ks = rng.uniform(0.001, 0.01, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.001, 0.01, (nb, hkv)).astype(np.float32)
    bt = np.array([[3, 0, 4, np.iinfo(np.int32).max]], np.int32)
    q = _bf16(rng, (ql, hq, d))
    out, lse = oracle.attention(codes_k, codes_v, q, np.array([0, ql], np.int32),
                                np.array([L], np.int32), bt, 0.25,
                                k_scale=ks, v_scale=vs, lib=lib)
    val = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    K = np.zeros((L, hkv, d))
    V = np.zeros((L, hkv, d))
    for p in range(L):
        b = bt[0, p // bs]
        K[p] = val[codes_k[b, :, p % bs]] * ks[b][:, None]
        V[p] = val[codes_v[b, :, p % bs]] * vs[b][:, None]
    qq = torch.from_numpy(_f64(q)).permute(1, 0, 2)
    kk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(2, 0)
    vv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(2, 0)
    pos = torch.arange(ql)[:, None] + (L - ql)
    mask = torch.arange(L)[None, :] <= pos
    ref = torch.nn.functional.scaled_dot_product_attention(
        qq[None], kk[None], vv[None], attn_mask=mask[None, None], scale=0.25)[0]
    ref = ref.permute(1, 0, 2).reshape(-1, d).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---- NVFP4 ---------------------------------------------------------------------

def e2m1_table() -> np.ndarray:
    """The 16 E2M1 values of the golden fixture (the published format table)."""
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "e2m1_values.txt")
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split("->")
                vals[int(c)] = float(v)
    assert sorted(vals) == list(range(16))
    return np.array([vals[c] for c in range(16)])


def _e2m1_nearest(x: float, table: np.ndarray) -> int:
    """Brute force: the code whose value is nearest to x (saturating beyond
    +-6), ties to the code with an even mantissa bit, zero keeps x's sign."""
    if math.isnan(x):
        return 0x8 if math.copysign(1.0, x) < 0 else 0x0
    cands = range(8, 16) if math.copysign(1.0, x) < 0 else range(0, 8)
    best = None
    for c in cands:
        dist = abs(x - table[c])
        key = (dist, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def pin_e2m1_decode(lib):
    """All 16 codes decode to the published E2M1 value table."""
    table = e2m1_table()
    for c in range(16):
        got = lib.pko_e2m1_value(c)
        assert got == table[c] and math.copysign(1.0, got) == math.copysign(1.0, table[c]), c


def pin_e2m1_encode(lib):
    """Encoding picks the nearest table value (brute force), ties to the even
    code, saturating at +-6; every table value encodes to its own code."""
    table = e2m1_table()
    enc = lib.pko_e2m1_encode
    for c in range(16):
        assert enc(float(table[c])) == c, c
    rng = np.random.default_rng(31)
    mids = [(table[c] + table[c + 1]) / 2 for c in range(7)]
    xs = np.concatenate([rng.uniform(-8, 8, 4000), rng.standard_normal(2000) * 2,
                         mids, [-m for m in mids], [5.0, -5.0, 6.0, 7.0, 1e9, -1e9,
                                                       0.25, 0.75, 2.5, 3.5]])
    for x in xs.astype(np.float32):
        assert enc(float(x)) == _e2m1_nearest(float(x), table), float(x)
    # ties: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert [enc(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == [0, 2, 2, 4, 4, 6, 6]
    assert enc(float("inf")) == 7 and enc(float("-inf")) == 15


def _nvfp4_reference_row(x_bits: np.ndarray, scale: np.float32, table: np.ndarray):
    """NVFP4 quantisation of one row with numpy fp32 arithmetic, torch's E4M3
    cast for the micro scale and brute-force nearest E2M1 codes."""
    d = x_bits.shape[0]
    x = _f64(x_bits).astype(np.float32)
    codes = np.zeros(d // 2, np.uint8)
    ms = np.zeros(d // 16, np.uint8)
    for b in range(d // 16):
        blk = x[16 * b:16 * b + 16]
        amax = np.float32(np.nanmax(np.abs(blk))) if not np.all(np.isnan(blk)) else np.float32(0)
        ratio = np.float32(amax / np.float32(np.float32(6.0) * scale))
        m = torch.tensor([min(float(ratio), 448.0)], dtype=torch.float32).to(
            torch.float8_e4m3fn)
        ms[b] = m.view(torch.uint8).item()
        msv = m.to(torch.float32).item()
        c = np.zeros(16, np.uint8)
        if msv != 0.0:
            step = np.float32(scale * np.float32(msv))
            for i in range(16):
                c[i] = _e2m1_nearest(float(np.float32(blk[i] / step)), table)
        codes[8 * b:8 * b + 8] = c[0::2] | (c[1::2] << 4)
    return codes, ms


def pin_nvfp4_quantize(lib):
    """NVFP4 row quantisation against an independent numpy/torch restatement
    (fp32 products and quotients, library E4M3 cast of the micro scale,
    brute-force nearest E2M1), on Gaussian rows, rows with outliers, rows
    whose micro scale saturates or underflows to zero, and an all-zero row."""
    table = e2m1_table()
    rng = np.random.default_rng(32)
    d = 128
    rows = [(_bf16(rng, (d,)), np.float32(2.2 / 2688)),
            (_bf16(rng, (d,), 40.0), np.float32(1e-3)),
            (_bf16(rng, (d,)), np.float32(1e-6)),      # micro scales saturate at 448
            (_bf16(rng, (d,), 1e-6), np.float32(1.0)),  # micro scales round to 0
            (np.zeros(d, np.uint16), np.float32(0.01))]
    spike = _bf16(rng, (d,))
    spike[5] = _bf16(rng, (1,), 300.0)[0]
    rows.append((spike, np.float32(0.004)))
    for x, sc in rows:
        codes, ms = _q(lib, x, sc)
        rc, rm = _nvfp4_reference_row(x, sc, table)
        assert np.array_equal(ms, rm)
        assert np.array_equal(codes, rc)


def _q(lib, x, sc):
    d = x.shape[0]
    codes = np.zeros(d // 2, np.uint8)
    ms = np.zeros(d // 16, np.uint8)
    lib.pko_nvfp4_quantize_row(np.ascontiguousarray(x, np.uint16), d, float(sc),
                               codes.ctypes.data_as(ctypes.c_void_p),
                               ms.ctypes.data_as(ctypes.c_void_p))
    return codes, ms


def nvfp4_split_tile(tile: np.ndarray, bs: int, d: int):
    """(codes [bs, d/2], micro scales [bs, d/16]) of one NVFP4 (block, KV
    head) tile: groups of min(bs, 64) rows, each its codes then its scales."""
    gs = min(bs, 64)
    per = gs * 9 * d // 16
    codes, ms = [], []
    for g0 in range(0, bs, gs):
        grp = tile[(g0 // gs) * per:(g0 // gs + 1) * per]
        codes.append(grp[:gs * d // 2].reshape(gs, d // 2))
        ms.append(grp[gs * d // 2:].reshape(gs, d // 16))
    return np.concatenate(codes), np.concatenate(ms)


def nvfp4_dequant_tile(tile: np.ndarray, bs: int, d: int, scale: float) -> np.ndarray:
    """[bs, d] values of one NVFP4 (block, KV head) tile; element 2j of a row
    is the low nibble of its code byte j."""
    table = e2m1_table()
    e4 = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    codes, ms = nvfp4_split_tile(tile, bs, d)
    nib = np.empty((bs, d), np.uint8)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    return table[nib] * np.repeat(e4[ms], 16, axis=1) * float(scale)


def pin_write_slots_nvfp4(lib):
    """NVFP4 append writes each new row's codes and micro scales (the row
    quantiser's output) at its slot inside the (block, KV head) tile and
    leaves every other byte alone."""
    for bs in (16, 128):
        _write_slots_nvfp4_case(lib, bs)


def _write_slots_nvfp4_case(lib, bs):
    rng = np.random.default_rng(33 + bs)
    nb, hkv, d = 4, 2, 128
    tile = bs * 9 * d // 16
    kc = np.full((nb, hkv, tile), 0xA5, np.uint8)
    vc = kc.copy()
    ks = rng.uniform(0.0005, 0.002, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.0005, 0.002, (nb, hkv)).astype(np.float32)
    T = 5
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[2] = -1
    kn = _bf16(rng, (T, hkv, d))
    vn = _bf16(rng, (T, hkv, d))
    k0, v0 = kc.copy(), vc.copy()
    oracle.write_slots(kc, vc, kn, vn, slots, k_scale=ks, v_scale=vs, lib=lib)
    table = e2m1_table()
    for cache, ref0, src, sc in ((kc, k0, kn, ks), (vc, v0, vn, vs)):
        want = ref0.copy()
        for t, s in enumerate(slots):
            if s < 0:
                continue
            b, o = s // bs, s % bs
            gs = min(bs, 64)
            base = (o // gs) * gs * 9 * d // 16
            r = o % gs
            for h in range(hkv):
                c, m = _nvfp4_reference_row(src[t, h], sc[b, h], table)
                want[b, h, base + r * d // 2:base + (r + 1) * d // 2] = c
                mb = base + gs * d // 2
                want[b, h, mb + r * d // 16:mb + (r + 1) * d // 16] = m
        assert np.array_equal(cache, want)


def pin_nvfp4_attention(lib):
    """NVFP4 pools attend over e2m1(code) * e4m3(micro scale) * scale: same
    result as fp64 SDPA over the tiles dequantised by the published E2M1
    table and torch's E4M3 decode."""
    for bs, L in ((8, 21), (128, 300)):
        _nvfp4_attention_case(lib, bs, L)


def _nvfp4_attention_case(lib, bs, L):
    rng = np.random.default_rng(34 + bs)
    hq, hkv, d = 4, 2, 32
    ql = 3
    nb = 5
    tile = bs * 9 * d // 16
    kc = rng.integers(0, 256, (nb, hkv, tile)).astype(np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, tile)).astype(np.uint8)
    # micro scales: finite E4M3 codes between 2^-3 and 2^4
    gs = min(bs, 64)
    per = gs * 9 * d // 16
    for c in (kc, vc):
        for g0 in range(0, bs, gs):
            base = (g0 // gs) * per + gs * d // 2
            c[:, :, base:base + gs * d // 16] = rng.integers(0x20, 0x58, (nb, hkv, gs * d // 16))
    ks = rng.uniform(0.05, 0.2, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.05, 0.2, (nb, hkv)).astype(np.float32)
    bt = np.array([[3, 0, 4, np.iinfo(np.int32).max]], np.int32)
    q = _bf16(rng, (ql, hq, d))
    out, lse = oracle.attention(kc, vc, q, np.array([0, ql], np.int32),
                                np.array([L], np.int32), bt, 0.25,
                                k_scale=ks, v_scale=vs, lib=lib)
    K = np.zeros((L, hkv, d))
    V = np.zeros((L, hkv, d))
    for p in range(L):
        b = bt[0, p // bs]
        for h in range(hkv):
            K[p, h] = nvfp4_dequant_tile(kc[b, h], bs, d, ks[b, h])[p % bs]
            V[p, h] = nvfp4_dequant_tile(vc[b, h], bs, d, vs[b, h])[p % bs]
    qq = torch.from_numpy(_f64(q)).permute(1, 0, 2)
    kk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(2, 0)
    vv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(2, 0)
    pos = torch.arange(ql)[:, None] + (L - ql)
    mask = torch.arange(L)[None, :] <= pos
    ref = torch.nn.functional.scaled_dot_product_attention(
        qq[None], kk[None], vv[None], attn_mask=mask[None, None], scale=0.25)[0]
    ref = ref.permute(1, 0, 2).reshape(-1, d).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


ALL_PINS = [pin_sdpa, pin_block_permutation, pin_chunked_prefill,
            pin_closed_forms, pin_gqa_is_repeated_mha, pin_lse_merge,
            pin_context_parallel_shards, pin_rope_is_a_complex_rotation, pin_bf16_round,
            pin_write_slots_bf16, pin_e4m3_decode, pin_e4m3_encode,
            pin_write_slots_fp8, pin_fp8_attention, pin_e2m1_decode, pin_e2m1_encode,
            pin_nvfp4_quantize, pin_write_slots_nvfp4, pin_nvfp4_attention]
