"""The host block pool (include/pkv_blocks.h) on CPU: the capacity rule and
prefix reuse of the pages, eviction order, slots, and a randomized
comparison with a small independent model of the same rules."""
import random

import numpy as np
import pytest

import paged_kv_attention_pkv_gb300 as pkv


def cdiv(a, b):
    return -(-a // b)


def test_capacity_does_not_count_hit_blocks_that_are_eviction_candidates():
    """Page "vLLM/V1 推理调度器", section 源码片段 (allocate_slots): hit blocks with
    no reference are free blocks too, so they cannot also pay for new ones."""
    bp = pkv.Blocks(4, 4)
    a = list(range(100, 112))                       # 12 tokens = 3 full blocks
    ta, nc = bp.allocate(1, a, 12)
    assert nc == 0 and len(ta) == 3
    bp.commit(1, a, 12)
    bp.free(1)
    assert bp.stats() == {"free": 4, "cached": 3, "evictable": 3}
    b = a + [7, 7, 7, 7, 7]                          # 17 tokens: 3 hit + 2 new blocks
    assert bp.lookup(b) == 12
    t, _ = bp.allocate(2, b, 17 - 12)
    assert t is None                                 # 2 new > 4 free - 3 evictable hits
    assert bp.stats() == {"free": 4, "cached": 3, "evictable": 3}   # nothing changed
    c = a + [7, 7, 7, 7]                             # 16 tokens: 3 hit + 1 new block
    tc, ncc = bp.allocate(3, c, 16 - 12)
    assert ncc == 12 and list(tc[:3]) == list(ta) and len(tc) == 4
    assert [bp.ref_count(x) for x in tc] == [1, 1, 1, 1]
    assert bp.stats()["free"] == 0


def test_shared_prefix_blocks_are_reused_and_counted():
    bp = pkv.Blocks(64, 16)
    prefix = list(range(48))                         # 3 full blocks
    a = prefix + [1000 + i for i in range(20)]
    ta, _ = bp.allocate(1, a, len(a))
    bp.commit(1, a, len(a))
    b = prefix + [2000 + i for i in range(5)]
    assert bp.lookup(b) == 48
    tb, ncb = bp.allocate(2, b, len(b) - 48)
    assert ncb == 48 and list(tb[:3]) == list(ta[:3]) and tb[3] not in ta
    assert [bp.ref_count(x) for x in ta[:3]] == [2, 2, 2]
    # an all-hit prompt still computes its last token
    assert bp.lookup(prefix) == 32
    bp.free(1)
    assert [bp.ref_count(x) for x in ta[:3]] == [1, 1, 1]
    bp.free(2)
    st = bp.stats()
    assert st["free"] == 64 and st["cached"] == 4 and st["evictable"] == 4


def test_least_recently_released_first_and_tail_before_head():
    bp = pkv.Blocks(6, 2)
    a = [1, 2, 3, 4, 5, 6]                           # 3 full blocks
    ta, _ = bp.allocate(1, a, 6)
    bp.commit(1, a, 6)
    bp.free(1)                                       # queue: 3 unused, then a2, a1, a0
    x, _ = bp.allocate(2, [9] * 6, 6)                # takes the 3 never-used blocks
    assert not set(x) & set(ta)
    y, _ = bp.allocate(3, [8, 8], 2)                 # next: A's tail block
    assert list(y) == [ta[2]]
    assert bp.lookup(a + [0]) == 4                   # its cache entry is gone
    assert bp.stats()["cached"] == 2


def test_decode_growth_and_slots():
    bp = pkv.Blocks(16, 4)
    toks = [5, 6, 7]
    t, nc = bp.allocate(1, toks, 3)
    assert nc == 0 and len(t) == 1
    bp.commit(1, toks, 3)
    for step in range(6):                            # decode: one new token per step
        toks = toks + [10 + step]
        t, nc = bp.allocate(1, toks, 1)
        assert nc == len(toks) - 1 and len(t) == cdiv(len(toks), 4)
        bp.commit(1, toks, len(toks))
    s = bp.slots(1, 0, len(toks))
    assert list(s) == [int(t[p // 4]) * 4 + p % 4 for p in range(len(toks))]
    with pytest.raises(pkv.PkvError):
        bp.slots(1, 0, len(t) * 4 + 1)               # past the table
    with pytest.raises(pkv.PkvError):
        bp.free(99)                                  # unknown request


def test_lookahead_blocks_are_reserved():
    bp = pkv.Blocks(8, 4)
    t, _ = bp.allocate(1, [1, 2, 3, 4], 4, num_lookahead=3)
    assert len(t) == cdiv(4 + 3, 4)


# ---- randomized comparison with an independent model -------------------------

class Model:
    """The same rules, written plainly: a dict cache keyed by the tuple of
    all tokens up to and including a block, a list as the free queue."""

    def __init__(self, n, bs):
        self.bs = bs
        self.ref = [0] * n
        self.key = [None] * n           # cache key of a block, or None
        self.cache = {}                 # key -> block
        self.queue = list(range(n))     # free blocks, front = next to reuse
        self.reqs = {}                  # req -> [table, num_computed, committed]

    def hits(self, toks):
        out = []
        for i in range((len(toks) - 1) // self.bs if toks else 0):
            k = tuple(toks[:(i + 1) * self.bs])
            if k not in self.cache:
                break
            out.append(self.cache[k])
        return out

    def allocate(self, req, toks, n_new):
        fresh = req not in self.reqs
        hit = self.hits(toks) if fresh else []
        comp = len(hit) * self.bs if fresh else self.reqs[req][1]
        held = 0 if fresh else len(self.reqs[req][0])
        need = cdiv(comp + n_new, self.bs) - held - len(hit)
        if need > len(self.queue) - sum(1 for b in hit if self.ref[b] == 0):
            return None, None
        if fresh:
            self.reqs[req] = [[], comp, len(hit)]
        r = self.reqs[req]
        for b in hit:
            if self.ref[b] == 0:
                self.queue.remove(b)
            self.ref[b] += 1
            r[0].append(b)
        for _ in range(max(need, 0)):
            b = self.queue.pop(0)
            if self.key[b] is not None:
                del self.cache[self.key[b]]
                self.key[b] = None
            self.ref[b] = 1
            r[0].append(b)
        return list(r[0]), r[1]

    def commit(self, req, toks, n):
        r = self.reqs[req]
        r[1] = max(r[1], n)
        for i in range(r[2], r[1] // self.bs):
            k = tuple(toks[:(i + 1) * self.bs])
            b = r[0][i]
            if self.key[b] is None and k not in self.cache:
                self.key[b] = k
                self.cache[k] = b
        r[2] = max(r[2], r[1] // self.bs)

    def free(self, req):
        for b in reversed(self.reqs.pop(req)[0]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.queue.append(b)


@pytest.mark.parametrize("seed", range(6))
def test_matches_an_independent_model(seed):
    rnd = random.Random(seed)
    n, bs = rnd.choice([(24, 4), (40, 2), (16, 8)])
    bp, md = pkv.Blocks(n, bs), Model(n, bs)
    prefixes = [[rnd.randrange(50) for _ in range(rnd.randrange(1, 30))] for _ in range(3)]
    live = {}
    for step in range(300):
        op = rnd.random()
        if op < 0.45 and len(live) < 6:
            req = step
            toks = rnd.choice(prefixes) + [rnd.randrange(50) for _ in range(rnd.randrange(0, 12))]
            if not toks:
                continue
            assert bp.lookup(toks) == len(md.hits(toks)) * bs
            hit = len(md.hits(toks)) * bs
            n_new = rnd.randrange(1, len(toks) - hit + 1)
            t1, c1 = bp.allocate(req, toks, n_new)
            t2, c2 = md.allocate(req, toks, n_new)
            assert (None if t1 is None else list(t1)) == t2 and c1 == c2
            if t1 is not None:
                live[req] = [toks, c1 + n_new]
                bp.commit(req, toks, c1 + n_new)
                md.commit(req, toks, c1 + n_new)
        elif op < 0.75 and live:
            req = rnd.choice(sorted(live))
            toks, done = live[req]
            if done >= len(toks):
                toks = toks + [rnd.randrange(50)]
            t1, c1 = bp.allocate(req, toks, 1)
            t2, c2 = md.allocate(req, toks, 1)
            assert (None if t1 is None else list(t1)) == t2 and c1 == c2
            if t1 is not None:
                live[req] = [toks, done + 1]
                bp.commit(req, toks, done + 1)
                md.commit(req, toks, done + 1)
        elif live:
            req = rnd.choice(sorted(live))
            bp.free(req)
            md.free(req)
            del live[req]
        st = bp.stats()
        assert st["free"] == len(md.queue)
        assert st["cached"] == len(md.cache)
        assert all(bp.ref_count(b) == md.ref[b] for b in range(n))
