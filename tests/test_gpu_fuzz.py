"""Randomised small steps against the fp64 oracle (GPU only).

Each case draws a step at random from a fixed seed: the number of requests,
their new-token counts (decodes, short chunks on the decode kernel, prefill
rows on the tensor cores, few tiles whose key ranges get split), their
context lengths (block-aligned or not), the query group, the block size and
the pool format, with the handle's staging pools on or off.  Every output row
and its log-sum-exp are compared with the oracle, so interplays the
hand-picked sweeps do not name (a split prefill next to a staged one, chunked
decode rows beside split decode pairs, ...) are covered too.
"""
import numpy as np
import pytest

import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

N_CASES = 24


def draw(seed: int):
    rng = np.random.default_rng(1000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    kv = str(rng.choice(["bf16", "fp8", "nvfp4"]))
    B = int(rng.integers(1, 7))
    q_lens, seq_lens = [], []
    for _ in range(B):
        kind = rng.random()
        if kind < 0.4:
            q = 1                                   # decode
        elif kind < 0.6:
            q = int(rng.integers(2, 9))             # a few tokens
        else:
            q = int(rng.integers(9, 400))           # prefill rows
        hist = int(rng.integers(0, 6000))
        if rng.random() < 0.3:
            hist = hist // bs * bs                  # block-aligned history
        q_lens.append(q)
        seq_lens.append(hist + q)
    stage = bool(rng.random() < 0.7)
    q_scale = 8.0 if rng.random() < 0.25 else 1.0
    return (f"fuzz{seed}_{kv}_g{G}_bs{bs}", G * hkv, hkv, bs, q_lens, seq_lens, kv, stage,
            q_scale)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_step_every_row(seed):
    name, hq, hkv, bs, q_lens, seq_lens, kv, stage, q_scale = draw(seed)
    s = W.custom_spec(name, hq, hkv, bs, q_lens, seq_lens, seed=seed, kv_dtype=kv)
    b = W.generate(s, "cuda", q_scale=q_scale)
    U.full_parity(b, what=f"{name} q {q_lens} L {seq_lens} stage {stage}",
                  peaked=q_scale > 1.0, stage=stage)
