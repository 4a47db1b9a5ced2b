"""Seeded synthetic workloads for paged KV attention.

This module only builds inputs: sequence lengths, block tables, slot
mappings, KV pools, queries and new K/V rows.  It holds none of the attention
arithmetic, and both the oracle tests and the CUDA tests draw their inputs
from it.  The shapes follow the agentic workloads the pages describe; none of
the traces or datasets those pages measure on is reproduced (they are not
available here), only their published shapes:

* long, growing contexts with a shared sub-agent prefix of about 10K tokens
  and contexts up to ~141.5K ("vLLM Agentic 推理｜面向 Agent 负载的推理优化",
  sections 2.1 and 3.1: median input 142K, >96% prefix reuse);
* incremental prefill of l_incr new tokens over l_hist history ("AMPD：PD
  分离遇上多轮推理，incremental prefill 到底该在哪跑", sections 1 and 3);
* the per-step token budget and long-prefill threshold of the V1 scheduler
  and block counts num_required_blocks = cdiv(computed + new, block_size)
  ("vLLM/V1 推理调度器", section 源码片段).

Random streams: ``torch.Generator().manual_seed(seed * 16 + stream)`` with
stream 0 = lengths, 1 = block permutation, 2 = Q, 3 = K pool, 4 = V pool,
5 = new K, 6 = new V.  Large pools are drawn on the GPU from a CUDA generator
with the same seed; small ones on the CPU.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
BF16_NAN = 0x7FC0      # quiet-NaN bit pattern used as poison in bf16 pools
E4M3_NAN = 0x7F        # NaN code of E4M3 (S.1111.111) used as poison in FP8 pools
E4M3_MAX = 448.0

S_LEN, S_PERM, S_Q, S_K, S_V, S_KNEW, S_VNEW = range(7)


def cdiv(a: int, b: int) -> int:
    """Ceiling division, the block count rule of the V1 KV-cache manager."""
    return -(-a // b)


def schedule_step(num_decodes: int, prefill_needs: list[int], threshold: int,
                  budget: int, max_model_len: int | None = None,
                  computed: list[int] | None = None) -> list[int]:
    """Token counts the V1 scheduler grants the prefills of one step.

    Running decodes are served first (one token each); every prefill then
    gets min(need, threshold, remaining budget, max_model_len - computed)
    tokens, in order, until the budget is spent ("vLLM/V1 推理调度器",
    section 处理流程 steps 1-2 and the Scheduler.schedule token-budget code).
    """
    left = budget - num_decodes
    out = []
    for i, need in enumerate(prefill_needs):
        n = need
        if 0 < threshold < n:
            n = threshold
        n = min(n, left)
        if max_model_len is not None:
            n = min(n, max_model_len - (computed[i] if computed else 0))
        if n <= 0:
            break
        out.append(n)
        left -= n
    return out


@dataclass
class Spec:
    """Shape of one workload (lengths already drawn)."""
    name: str
    hq: int
    hkv: int
    block_size: int
    kv_dtype: str                      # "bf16", "fp8" or "nvfp4"
    q_lens: list[int]
    seq_lens: list[int]
    seed: int
    shared_prefix: tuple[list[int], int] | None = None   # (seq ids, tokens)
    pool_blocks: int | None = None     # fixed pool size, else needed + 5 %
    head_dim: int = HEAD_DIM

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_lens))


def _gen(seed: int, stream: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + stream)
    return g


def _uniform_int(g: torch.Generator, lo: int, hi: int, n: int) -> list[int]:
    """n integers uniform in [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def _lognormal_int(g: torch.Generator, median: float, sigma: float, lo: int,
                   hi: int, n: int) -> list[int]:
    z = torch.randn((n,), generator=g, dtype=torch.float64)
    vals = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return [int(v) for v in vals.tolist()]


CONFIG_NAMES = ["c1_tiny_prefill", "c2_decode", "c3_post_tool_prefill",
                "c4_mixed_step", "c5_fp8_long_decode"]

# Prefill needs behind the mixed step: two long prompts, two ~1K and three
# ~0.5K tool results, one more long prompt that the budget truncates.
C4_PREFILL_NEEDS = [4096, 4096, 1024, 1024, 512, 512, 512, 4096]


def config_spec(index: int) -> Spec:
    """The five benchmark workloads, index 0..4, with lengths drawn."""
    seed = 1000 + index
    g = _gen(seed, S_LEN)
    if index == 0:
        # 1 sequence, l_hist 1000 + l_incr 64, 8q/2kv heads, 128-block pool
        return Spec(CONFIG_NAMES[0], 8, 2, 16, "bf16", [64], [1064], seed,
                    pool_blocks=128)
    if index == 1:
        lens = _uniform_int(g, 4096, 32768, 64)
        return Spec(CONFIG_NAMES[1], 32, 8, 16, "bf16", [1] * 64, lens, seed)
    if index == 2:
        hist = _lognormal_int(g, 48000, 0.5, 10000, 141000, 16)
        incr = _uniform_int(g, 200, 3000, 16)
        lens = [h + q for h, q in zip(hist, incr)]
        return Spec(CONFIG_NAMES[2], 32, 8, 16, "bf16", incr, lens, seed,
                    shared_prefix=([0, 1, 2, 3], 10000))
    if index == 3:
        dec = _uniform_int(g, 30000, 140000, 120)
        chunks = schedule_step(120, C4_PREFILL_NEEDS, 2048, 8192)
        hist = _lognormal_int(g, 142000, 0.5, 60000, 200000, len(chunks))
        q_lens = [1] * 120 + chunks
        lens = dec + [h + q for h, q in zip(hist, chunks)]
        return Spec(CONFIG_NAMES[3], 64, 8, 16, "bf16", q_lens, lens, seed)
    if index == 4:
        lens = _uniform_int(g, 524288, 1048576, 8)
        return Spec(CONFIG_NAMES[4], 64, 8, 64, "fp8", [1] * 8, lens, seed)
    raise ValueError(index)


@dataclass
class Batch:
    """One step's inputs.  Host metadata is numpy; tensors live on ``device``."""
    spec: Spec
    qsl: np.ndarray              # [B+1] int32
    seq_lens: np.ndarray         # [B] int32
    block_tables: np.ndarray     # [B, stride] int32
    slot_mapping: np.ndarray     # [T] int64
    num_blocks: int
    poison_block: int            # an unused block id filled with NaN poison
    q: torch.Tensor              # [T, Hq, D] bf16
    k_new: torch.Tensor          # [T, Hkv, D] bf16
    v_new: torch.Tensor
    k_cache: torch.Tensor        # [NB, Hkv, bs, D] bf16 or uint8
    v_cache: torch.Tensor
    k_scale: torch.Tensor | None = None   # [NB, Hkv] float32 (fp8 only)
    v_scale: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.qsl[-1])


def _layout(spec: Spec, perm_gen: torch.Generator, tail_entries: int):
    """Assign physical block ids: shared prefixes reuse the same ids."""
    bs = spec.block_size
    nblk = [cdiv(L, bs) for L in spec.seq_lens]
    shared_ids, shared_n = ([], 0)
    if spec.shared_prefix is not None:
        shared_ids, shared_tok = spec.shared_prefix
        assert shared_tok % bs == 0, "sharing is of whole blocks only"
        shared_n = shared_tok // bs
        for s in shared_ids:
            assert spec.seq_lens[s] - spec.q_lens[s] >= shared_tok
    needed = sum(nblk) - shared_n * max(0, len(shared_ids) - 1)
    pool = spec.pool_blocks or (needed + cdiv(needed * 5, 100) + 1)
    assert pool >= needed + 1, "pool too small"
    perm = torch.randperm(pool, generator=perm_gen).numpy().astype(np.int64)
    stride = max(nblk) + tail_entries
    tables = np.zeros((spec.num_seqs, stride), dtype=np.int64)
    nxt = 0
    shared_block_ids = None
    for i, n in enumerate(nblk):
        start = 0
        if i in shared_ids:
            if shared_block_ids is None:
                shared_block_ids = perm[nxt:nxt + shared_n].copy()
                nxt += shared_n
            tables[i, :shared_n] = shared_block_ids
            start = shared_n
        tables[i, start:n] = perm[nxt:nxt + (n - start)]
        nxt += n - start
    assert nxt == needed
    poison_block = int(perm[needed])
    used = perm[:needed]
    return tables, nblk, pool, poison_block, used


def _fill_normal(t: torch.Tensor, g: torch.Generator, chunk_rows: int = 1 << 20,
                 sigma: float = 1.0):
    """Fill a [rows, D] view with N(0, sigma^2) in chunks (bounded temporaries)."""
    rows = t.shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        t[r0:r1] = (torch.randn((r1 - r0, t.shape[1]), generator=g, device=t.device,
                                dtype=torch.float32) * sigma).to(t.dtype)


def _fill_fp8_pool(codes: torch.Tensor, scales: torch.Tensor, g: torch.Generator,
                   chunk_blocks: int = 2048, sigma: float = 1.0):
    """E4M3 pool from an N(0, sigma^2) source, one fp32 scale per (block, KV
    head): scale = amax/448 over the block, codes = source/scale cast to E4M3
    by torch (a generator choice; the oracle reads the stored codes)."""
    nb, hkv, bs, d = codes.shape
    for b0 in range(0, nb, chunk_blocks):
        b1 = min(nb, b0 + chunk_blocks)
        src = torch.randn((b1 - b0, hkv, bs, d), generator=g,
                          device=codes.device, dtype=torch.float32) * sigma
        amax = src.abs().amax(dim=(2, 3))
        sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        q = (src / sc[:, :, None, None]).clamp(-E4M3_MAX, E4M3_MAX)
        codes[b0:b1] = q.to(torch.float8_e4m3fn).view(torch.uint8)
        scales[b0:b1] = sc


# NVFP4 pools: rows of 64 code bytes + 8 micro-scale bytes, grouped per
# min(block_size, 64) rows inside a (block, KV head) tile.
NVFP4_ROW = 72
NVFP4_GROUP = 64
# magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 drawn with roughly the frequencies a
# Gaussian block quantised against its own largest element shows
_E2M1_MAG_WEIGHTS = [0.06, 0.12, 0.115, 0.11, 0.147, 0.16, 0.158, 0.13]


def nvfp4_row_bytes(bs: int, off: np.ndarray, head_dim: int = HEAD_DIM):
    """Byte positions inside an NVFP4 (block, KV head) tile of the codes
    ([n, D/2]) and micro scales ([n, D/16]) of rows `off`."""
    gs = min(bs, NVFP4_GROUP)
    off = np.asarray(off, dtype=np.int64)
    base = (off // gs) * gs * (head_dim // 2 + head_dim // 16)
    r = off % gs
    codes = base[:, None] + r[:, None] * (head_dim // 2) + np.arange(head_dim // 2)[None, :]
    ms = (base[:, None] + gs * (head_dim // 2) + r[:, None] * (head_dim // 16) +
          np.arange(head_dim // 16)[None, :])
    return codes, ms


def _fill_nvfp4_pool(tiles: torch.Tensor, scales: torch.Tensor, g: torch.Generator,
                     chunk_blocks: int = 2048, sigma: float = 1.0):
    """NVFP4 tiles drawn directly as codes (no quantisation here): E2M1
    nibbles with Gaussian-like magnitude frequencies and random signs; micro
    scales the E4M3 codes (torch's cast) of U[1, 3] / (6 scale); the (block,
    KV head) scale sigma * U[3.5, 4.5] / 2688, so that values look like a
    N(0, sigma^2) source quantised the usual way."""
    nb, hkv, tb = tiles.shape
    bs = tb // NVFP4_ROW
    gs = min(bs, NVFP4_GROUP)
    w = torch.tensor(_E2M1_MAG_WEIGHTS, dtype=torch.float32, device=tiles.device)
    for b0 in range(0, nb, chunk_blocks):
        b1 = min(nb, b0 + chunk_blocks)
        n = b1 - b0
        sc = (torch.rand((n, hkv), generator=g, device=tiles.device) + 3.5) / 2688.0
        mag = torch.multinomial(w, n * hkv * bs * 128, replacement=True, generator=g)
        sign = torch.randint(0, 2, mag.shape, generator=g, device=tiles.device) * 8
        nib = (mag + sign).to(torch.uint8).view(n, hkv, bs // gs, gs, 64, 2)
        codes = nib[..., 0] | (nib[..., 1] << 4)
        target = (torch.rand((n, hkv, bs // gs, gs, 8), generator=g, device=tiles.device) * 2 + 1)
        target = target / (6.0 * sc[:, :, None, None, None])
        ms = target.clamp(max=448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        grp = tiles[b0:b1].view(n, hkv, bs // gs, gs * NVFP4_ROW)
        grp[..., :gs * 64] = codes.reshape(n, hkv, bs // gs, gs * 64)
        grp[..., gs * 64:] = ms.reshape(n, hkv, bs // gs, gs * 8)
        scales[b0:b1] = sc * sigma


def generate(spec: Spec, device: str | torch.device = "cpu", q_scale: float = 1.0,
             tail_entries: int = 3, tail_fill: str = "poison_block",
             unused_poison: bool = True, kv_sigma: float = 1.0) -> Batch:
    """Build one step's inputs for ``spec``.

    K and V (pools and new rows) are drawn with standard deviation
    ``kv_sigma`` (quantised pools: their block scales follow), queries with
    ``q_scale``.

    History rows hold N(0,1) data; the rows of this step's new tokens and the
    rows past each sequence's end hold NaN poison until ``write_slots`` fills
    the new ones.  Block-table entries past cdiv(L, bs) hold ``poison_block``
    (a valid, NaN-filled block: reading it would show up as NaN, not as a
    fault) or, with ``tail_fill="int_max"``, INT32_MAX (CPU oracle tests).
    """
    device = torch.device(device)
    bs, hkv, hq, d = spec.block_size, spec.hkv, spec.hq, spec.head_dim
    gdev = "cuda" if device.type == "cuda" else "cpu"
    tables, nblk, pool, poison_block, used = _layout(
        spec, _gen(spec.seed, S_PERM), tail_entries)
    B = spec.num_seqs
    for i in range(B):
        fill = poison_block if tail_fill == "poison_block" else np.iinfo(np.int32).max
        tables[i, nblk[i]:] = fill
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(spec.q_lens)
    T = int(qsl[-1])
    seq_lens = np.asarray(spec.seq_lens, dtype=np.int32)
    # slots of the new tokens: logical position p = l_hist + t of sequence i
    slots = np.empty(T, dtype=np.int64)
    for i in range(B):
        h = spec.seq_lens[i] - spec.q_lens[i]
        p = np.arange(h, spec.seq_lens[i], dtype=np.int64)
        slots[qsl[i]:qsl[i + 1]] = tables[i, p // bs] * bs + p % bs

    fp8 = spec.kv_dtype == "fp8"
    nvfp4 = spec.kv_dtype == "nvfp4"
    cache_dtype = torch.uint8 if (fp8 or nvfp4) else torch.bfloat16
    shape = (pool, hkv, bs * NVFP4_ROW) if nvfp4 else (pool, hkv, bs, d)
    k_cache = torch.empty(shape, dtype=cache_dtype, device=device)
    v_cache = torch.empty_like(k_cache)
    k_scale = v_scale = None
    if nvfp4:
        k_scale = torch.empty((pool, hkv), dtype=torch.float32, device=device)
        v_scale = torch.empty_like(k_scale)
        _fill_nvfp4_pool(k_cache, k_scale, _gen(spec.seed, S_K, gdev), sigma=kv_sigma)
        _fill_nvfp4_pool(v_cache, v_scale, _gen(spec.seed, S_V, gdev), sigma=kv_sigma)
    elif fp8:
        k_scale = torch.empty((pool, hkv), dtype=torch.float32, device=device)
        v_scale = torch.empty_like(k_scale)
        _fill_fp8_pool(k_cache, k_scale, _gen(spec.seed, S_K, gdev), sigma=kv_sigma)
        _fill_fp8_pool(v_cache, v_scale, _gen(spec.seed, S_V, gdev), sigma=kv_sigma)
    else:
        _fill_normal(k_cache.view(-1, d), _gen(spec.seed, S_K, gdev), sigma=kv_sigma)
        _fill_normal(v_cache.view(-1, d), _gen(spec.seed, S_V, gdev), sigma=kv_sigma)

    def poison(cache, rows_blk, rows_off):
        if nvfp4:
            # codes 6, micro scales NaN: any read shows up as NaN
            ci, mi = nvfp4_row_bytes(bs, rows_off.cpu().numpy())
            rb = rows_blk[:, None]
            cache[rb, :, torch.as_tensor(ci, device=cache.device)] = 0x77
            cache[rb, :, torch.as_tensor(mi, device=cache.device)] = E4M3_NAN
            return
        if fp8:
            cache[rows_blk, :, rows_off, :] = E4M3_NAN
        else:
            cache.view(torch.int16)[rows_blk, :, rows_off, :] = BF16_NAN

    # unused blocks
    if unused_poison:
        mask = np.ones(pool, dtype=bool)
        mask[used] = False
        unused = torch.from_numpy(np.nonzero(mask)[0]).to(device)
        for cache in (k_cache, v_cache):
            if fp8 or nvfp4:
                cache[unused] = E4M3_NAN
            else:
                cache.view(torch.int16)[unused] = BF16_NAN
        if fp8 or nvfp4:
            k_scale[unused] = 1.0
            v_scale[unused] = 1.0
    # rows past the end of each sequence's last block
    tb, to = [], []
    for i in range(B):
        L = spec.seq_lens[i]
        last = tables[i, nblk[i] - 1]
        for off in range(L - (nblk[i] - 1) * bs, bs):
            tb.append(last)
            to.append(off)
    # rows of this step's new tokens
    tb.extend((slots // bs).tolist())
    to.extend((slots % bs).tolist())
    if tb:
        rb = torch.as_tensor(tb, dtype=torch.int64, device=device)
        ro = torch.as_tensor(to, dtype=torch.int64, device=device)
        poison(k_cache, rb, ro)
        poison(v_cache, rb, ro)

    gq = _gen(spec.seed, S_Q, gdev)
    q = (torch.randn((T, hq, d), generator=gq, device=device) * q_scale).to(torch.bfloat16)
    k_new = (torch.randn((T, hkv, d), generator=_gen(spec.seed, S_KNEW, gdev),
                         device=device) * kv_sigma).to(torch.bfloat16)
    v_new = (torch.randn((T, hkv, d), generator=_gen(spec.seed, S_VNEW, gdev),
                         device=device) * kv_sigma).to(torch.bfloat16)
    return Batch(spec, qsl, seq_lens, tables.astype(np.int32), slots, pool,
                 poison_block, q, k_new, v_new, k_cache, v_cache, k_scale,
                 v_scale)


def custom_spec(name: str, hq: int, hkv: int, block_size: int, q_lens, seq_lens,
                seed: int = 7, kv_dtype: str = "bf16", pool_blocks=None,
                shared_prefix=None) -> Spec:
    return Spec(name, hq, hkv, block_size, kv_dtype, list(q_lens),
                list(seq_lens), seed, shared_prefix=shared_prefix,
                pool_blocks=pool_blocks)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_pool(batch: Batch, which: str) -> np.ndarray:
    """Host copy of a pool as raw bits (uint16 for bf16, uint8 for E4M3)."""
    c = batch.k_cache if which == "k" else batch.v_cache
    if c.dtype == torch.uint8:
        return c.contiguous().cpu().numpy()
    return bf16_bits(c)


def subset(batch: Batch, seq_ids: list[int], kv_heads: list[int] | None = None):
    """Host inputs restricted to some sequences and KV heads, for sampled
    oracle checks at full size.

    Returns a dict of numpy arrays: a compact pool holding only the blocks the
    chosen sequences reference (renumbered; attention does not depend on
    physical ids) and only the chosen KV heads, their block tables, lengths,
    the query rows of those heads' groups, the new K/V rows, and the slots of
    those new rows in the compact pool.  Call it before the append so the
    pools still hold the generator's contents.  All query tokens of the
    chosen sequences are kept (positions depend on the token count); pick
    rows to evaluate with the oracle's ``rows`` argument.
    """
    spec = batch.spec
    bs = spec.block_size
    G = spec.hq // spec.hkv
    kvh = list(range(spec.hkv)) if kv_heads is None else list(kv_heads)
    heads = [h * G + g for h in kvh for g in range(G)]
    kc, vc = batch.k_cache, batch.v_cache
    ids = []
    for i in seq_ids:
        ids.extend(batch.block_tables[i, :cdiv(int(batch.seq_lens[i]), bs)].tolist())
    uniq = sorted(set(ids))
    remap = {b: j for j, b in enumerate(uniq)}
    dev = kc.device
    idx = torch.as_tensor(uniq, dtype=torch.int64, device=dev)
    hidx = torch.as_tensor(kvh, dtype=torch.int64, device=dev)

    def take(c):
        sub = c.index_select(0, idx).index_select(1, hidx).contiguous()
        if sub.dtype == torch.uint8:
            return sub.cpu().numpy()
        return bf16_bits(sub)

    nb = [cdiv(int(batch.seq_lens[i]), bs) for i in seq_ids]
    bt = np.zeros((len(seq_ids), max(nb)), dtype=np.int32)
    qsl = [0]
    tok = []
    slots = []
    for r, i in enumerate(seq_ids):
        bt[r, :nb[r]] = [remap[b] for b in batch.block_tables[i, :nb[r]].tolist()]
        a, b = int(batch.qsl[i]), int(batch.qsl[i + 1])
        tok.extend(range(a, b))
        qsl.append(qsl[-1] + (b - a))
        for s in batch.slot_mapping[a:b].tolist():
            slots.append(remap[s // bs] * bs + s % bs)
    qt = torch.as_tensor(tok, dtype=torch.int64, device=batch.q.device)
    hq_idx = torch.as_tensor(heads, dtype=torch.int64, device=batch.q.device)
    out = {
        "k_cache": take(kc), "v_cache": take(vc),
        "block_tables": bt, "seq_lens": batch.seq_lens[seq_ids].astype(np.int32),
        "qsl": np.asarray(qsl, dtype=np.int32),
        "q": bf16_bits(batch.q.index_select(0, qt).index_select(1, hq_idx)),
        "k_new": bf16_bits(batch.k_new.index_select(0, qt).index_select(1, hidx)),
        "v_new": bf16_bits(batch.v_new.index_select(0, qt).index_select(1, hidx)),
        "slot_mapping": np.asarray(slots, dtype=np.int64),
        "tokens": np.asarray(tok, dtype=np.int64),
        "heads": np.asarray(heads, dtype=np.int64),
    }
    if batch.k_scale is not None:
        out["k_scale"] = batch.k_scale.index_select(0, idx).index_select(1, hidx).cpu().numpy()
        out["v_scale"] = batch.v_scale.index_select(0, idx).index_select(1, hidx).cpu().numpy()
    return out


def algorithmic_work(spec: Spec) -> dict:
    """Bytes and flops the method must move / compute for one step.

    decode bytes: every context token's K and V rows once, plus Q and O;
    append bytes: read + write of the new K/V rows;
    prefill flops: 4 * D * Hq per causal (query, key) pair.
    """
    d, hq, hkv, bs = spec.head_dim, spec.hq, spec.hkv, spec.block_size
    # bytes per stored element (NVFP4: codes and micro scales, 72 per 128)
    s = {"fp8": 1, "nvfp4": NVFP4_ROW / 128}.get(spec.kv_dtype, 2)
    dec_bytes = 0
    pre_flops = 0
    pre_bytes = 0
    n_dec = n_pre = 0
    for q, L in zip(spec.q_lens, spec.seq_lens):
        h = L - q
        if q * (hq // hkv) <= 8:
            n_dec += 1
            dec_bytes += int(L * 2 * hkv * d * s) + 2 * q * hq * d * 2
            if s != 2:
                dec_bytes += cdiv(L, bs) * hkv * 2 * 4
        else:
            n_pre += 1
            pre_flops += 4 * d * hq * (q * h + q * (q + 1) // 2)
            pre_bytes += int(L * 2 * hkv * d * s) + 2 * q * hq * d * 2
    T = spec.num_tokens
    append_bytes = int(T * 2 * hkv * d * (2 + s))
    return {"decode_bytes": dec_bytes, "prefill_flops": pre_flops,
            "prefill_bytes": pre_bytes, "append_bytes": append_bytes,
            "num_decode": n_dec, "num_prefill": n_pre}
