"""Block tables and slots from the host block pool drive the kernels:
a prefix shared through the cache is written once and read by every request
that hits it (GPU, against the oracle over the same pool and tables)."""
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
HQ, HKV, D, BS, NB = 32, 8, 128, 16, 64


def kv_rows(tokens, pos0, seed):
    """K or V rows of tokens at positions pos0.. (a function of token and
    position only, so equal prefixes give equal rows)."""
    out = np.empty((len(tokens), HKV, D), np.float32)
    for i, t in enumerate(tokens):
        g = np.random.default_rng([seed, int(t), pos0 + i])
        out[i] = g.standard_normal((HKV, D))
    return torch.from_numpy(out).to(torch.bfloat16)


KV_DTYPES = {"bf16": pkv.KV_BF16, "fp8": pkv.KV_FP8_E4M3, "nvfp4": pkv.KV_NVFP4}


@pytest.mark.parametrize("kv", ["bf16", "fp8", "nvfp4"])
def test_pool_tables_feed_prefill_prefix_hits_and_decode(kv):
    """Quantised pools run their prefill steps through the staging pools
    (each request stages the shared prefix blocks it reads)."""
    rng = np.random.default_rng(4)
    prefix = list(rng.integers(0, 1000, 100))
    reqs = {1: prefix + list(rng.integers(0, 1000, 37)),
            2: prefix + list(rng.integers(0, 1000, 21))}
    bp = pkv.Blocks(NB, BS)
    cfg = pkv.make_config(HQ, HKV, BS, NB, 4, 256, kv_dtype=KV_DTYPES[kv],
                          softmax_scale=1 / math.sqrt(D), flags=pkv.FLAG_VALIDATE,
                          stage_tokens=4 * 256)
    shape, dtype, scale_shape = pkv.pool_shapes(cfg)
    if kv == "bf16":
        kc = torch.full(shape, float("nan"), dtype=dtype, device=DEV)
        ks = vs = None
    else:
        # poison: NaN E4M3 codes / NVFP4 bytes whose micro scales are NaN
        kc = torch.full(shape, 0x7F if kv == "fp8" else 0xFF, dtype=dtype, device=DEV)
        # block scales of N(0, 1) rows, varying from block to block
        g = torch.Generator().manual_seed(5)
        ks = (0.006 + 0.01 * torch.rand(scale_shape, generator=g)).to(DEV)
        vs = (0.006 + 0.01 * torch.rand(scale_shape, generator=g)).to(DEV)
    vc = kc.clone()
    h = pkv.Handle(cfg)
    done = {}

    def step(batch):
        """batch: [(req, tokens, n_new)] -> attention over the new tokens."""
        tables, qsl, lens, slots, knew, vnew, qs = [], [0], [], [], [], [], []
        for req, toks, n_new in batch:
            t, comp = bp.allocate(req, toks, n_new)
            assert t is not None
            pos0 = comp if req not in done else done[req]
            assert pos0 + n_new == len(toks)
            tables.append(t)
            slots.append(bp.slots(req, pos0, n_new))
            new = toks[pos0:]
            knew.append(kv_rows(new, pos0, 1))
            vnew.append(kv_rows(new, pos0, 2))
            qs.append(kv_rows(new, pos0, 3).repeat_interleave(HQ // HKV, dim=1))
            qsl.append(qsl[-1] + n_new)
            lens.append(len(toks))
        stride = max(len(t) for t in tables) + 1
        bt = np.full((len(batch), stride), np.iinfo(np.int32).max, np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        qsl = np.array(qsl, np.int32)
        lens = np.array(lens, np.int32)
        q = torch.cat(qs).to(DEV)
        kn, vn = torch.cat(knew).to(DEV), torch.cat(vnew).to(DEV)
        sl = torch.from_numpy(np.concatenate(slots)).to(DEV)
        if kv == "bf16":
            kc0 = kc.view(torch.int16).cpu().numpy().view(np.uint16).copy()
            vc0 = vc.view(torch.int16).cpu().numpy().view(np.uint16).copy()
            ks0 = vs0 = None
        else:
            kc0, vc0 = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
            ks0, vs0 = ks.cpu().numpy(), vs.cpu().numpy()
        h.write_slots(kn, vn, sl, kc, vc, ks, vs)
        out, lse = h.attention_varlen(q, kc, vc, torch.from_numpy(qsl).to(DEV),
                                      torch.from_numpy(lens).to(DEV),
                                      torch.from_numpy(bt).to(DEV), qsl, lens,
                                      lse=torch.empty(q.shape[:2], dtype=torch.float32,
                                                      device=DEV),
                                      k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        h.check_device_errors()
        for req, toks, _ in batch:
            bp.commit(req, toks, len(toks))
            done[req] = len(toks)
        # oracle: its own append into the pool as it was, then attention
        oracle.write_slots(kc0, vc0, W.bf16_bits(kn), W.bf16_bits(vn),
                           np.concatenate(slots), ks0, vs0)
        ref, ref_lse = oracle.attention(kc0, vc0, W.bf16_bits(q), qsl, lens, bt,
                                        1 / math.sqrt(D), ks0, vs0)
        got = out.double().cpu().numpy().reshape(-1, D)
        got_lse = lse.double().cpu().numpy().reshape(-1)
        U.check(got, ref, got_lse, ref_lse, kv, f"pool-driven step ({kv})", scaled=True)
        return tables

    t1 = step([(1, reqs[1], len(reqs[1]))])                  # prefill of request 1
    assert bp.lookup(reqs[2]) == 96                          # 6 full blocks of the prefix
    t2 = step([(2, reqs[2], len(reqs[2]) - 96)])             # incremental prefill over the hit
    assert list(t2[0][:6]) == list(t1[0][:6])
    assert all(bp.ref_count(b) == 2 for b in t1[0][:6])
    for _ in range(3):                                       # decode both together
        reqs[1] = reqs[1] + [int(rng.integers(0, 1000))]
        reqs[2] = reqs[2] + [int(rng.integers(0, 1000))]
        step([(1, reqs[1], 1), (2, reqs[2], 1)])
    bp.free(1)
    bp.free(2)
    assert bp.stats()["free"] == NB
    h.close()
