"""Degenerate and boundary steps through the C ABI (GPU): the largest block
size, an empty step, requests with no new token in a batch, single-key
contexts, a whole batch of one-token prefills, and a step whose shapes are
exactly the handle's maxima."""
import numpy as np
import pytest
import torch

import paged_kv_attention_pkv_gb300 as pkv
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda"


def spec(name, hq, hkv, bs, q_lens, seq_lens, kv="bf16", seed=17):
    return W.custom_spec(name, hq, hkv, bs, q_lens, seq_lens, seed=seed, kv_dtype=kv)


@pytest.mark.parametrize("kv", ["bf16", "fp8", "nvfp4"])
def test_block_size_256(kv):
    """The largest blocks (NVFP4: four 64-row groups per block), with a
    300-token prefill (tensor-core tiles for bf16, 8-row decode-kernel
    chunks otherwise)."""
    b = W.generate(spec(f"bs256_{kv}", 32, 8, 256, [1, 1, 300], [255, 1000, 900], kv=kv), DEV)
    U.full_parity(b, what=f"bs256 {kv}")


def test_requests_with_no_new_token_are_skipped():
    """q_i = 0 requests own no output row and must not disturb the others."""
    b = W.generate(spec("q0", 32, 8, 16, [1, 0, 37, 0, 1], [100, 50, 400, 1, 1]), DEV)
    U.full_parity(b, what="q0")


def test_single_key_contexts_return_that_value():
    """L = 1: the output is the one V row (exactly, after bf16 rounding) and
    the lse is the one score."""
    b = W.generate(spec("one_key", 8, 2, 16, [1, 1, 1], [1, 1, 1]), DEV)
    out, lse = U.gpu_step(b)
    sub = W.subset(b, [0, 1, 2])
    v = torch.from_numpy(sub["v_new"].view(np.int16)).view(torch.bfloat16).to(DEV)
    G = 4
    assert torch.equal(out, v.repeat_interleave(G, dim=1))


def test_empty_step_is_a_no_op():
    b = W.generate(spec("empty_ref", 8, 2, 16, [3], [10]), DEV)
    h = U.make_handle(b)
    empty_i32 = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(q)
    h.attention_varlen(q, b.k_cache, b.v_cache, empty_i32, empty_i32,
                       torch.zeros((0, 1), dtype=torch.int32, device=DEV),
                       np.zeros(1, np.int32), np.zeros(0, np.int32), out=out)
    h.write_slots(q[:, :2], q[:, :2], torch.zeros(0, dtype=torch.int64, device=DEV),
                  b.k_cache, b.v_cache)
    torch.cuda.synchronize()
    h.check_device_errors()
    h.close()


def test_step_at_the_handle_maxima():
    """max_num_seqs and max_num_tokens exactly equal to the step's."""
    b = W.generate(spec("at_max", 64, 8, 16, [2, 1, 200], [3000, 17, 1500]), DEV)
    h = U.make_handle(b)
    assert h.config.max_num_seqs == 3 and h.config.max_num_tokens == 203
    out, lse = U.gpu_step(b, handle=h)
    sub = W.subset(b, [0, 1, 2])
    ref, ref_lse = U.oracle_subset(sub, b.spec)
    got, got_lse = U.gpu_rows(out, lse, sub)
    U.check(got, ref, got_lse, ref_lse, "bf16", "at_max", scaled=True)
    h.close()
