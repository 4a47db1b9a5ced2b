"""The fp64 oracle against library routines, closed forms and invariances
(CPU only).  See tests/pins.py for what each pin checks."""
import re
import os

import pytest

import workloads
from tests import pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def _golden_lines(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def test_scheduler_rules_golden():
    """cdiv block counts and the token-budget rule on hand-computed cases
    (page "vLLM/V1 推理调度器", section 源码片段)."""
    n = 0
    for line in _golden_lines("scheduler_rules.txt"):
        lhs, rhs = line.split("->")
        f = lhs.split()
        want = [int(x) for x in rhs.split()]
        if f[0] == "cdiv":
            comp, new, look, bs = map(int, f[1:])
            assert [workloads.cdiv(comp + new + look, bs)] == want, line
        elif f[0] == "budget":
            ndec, budget, thr = map(int, f[1:4])
            needs = [int(x) for x in f[4:]]
            assert workloads.schedule_step(ndec, needs, thr, budget) == want, line
        n += 1
    assert n >= 10


def test_mixed_step_composition():
    """The mixed step fills the 8192-token budget exactly: 120 decodes plus
    eight chunks capped at the 2048 long-prefill threshold."""
    s = workloads.config_spec(3)
    assert s.num_tokens == 8192
    assert s.q_lens[120:] == [2048, 2048, 1024, 1024, 512, 512, 512, 392]


def test_shared_prefix_layout():
    """Sub-agent sessions 0-3 reference the same 625 physical blocks."""
    s = workloads.config_spec(2)
    b = workloads.generate(workloads.custom_spec(
        "mini_shared", 4, 2, 16, [3, 2, 5], [10000 + 40, 10000 + 7, 10000 + 100],
        shared_prefix=([0, 1, 2], 10000)), "cpu")
    for i in (1, 2):
        assert (b.block_tables[i, :625] == b.block_tables[0, :625]).all()
    ids = set(b.block_tables[0, :626].tolist()) | set(b.block_tables[1, 625:626].tolist())
    assert len(ids) == 627
    assert s.shared_prefix == ([0, 1, 2, 3], 10000)
