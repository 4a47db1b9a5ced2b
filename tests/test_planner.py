"""Host planner (pkv_plan): work items cover every (request, KV head, row,
key) exactly as the causal definition needs, split partials are laid out for
the combine, and bad metadata is rejected (CPU only)."""
import numpy as np
import pytest

import paged_kv_attention_pkv_gb300 as pkv
import workloads


def _plan(spec, num_sms=152):
    cfg = pkv.make_config(spec.hq, spec.hkv, spec.block_size, 10 ** 6,
                          max(1, spec.num_seqs), max(1, spec.num_tokens),
                          kv_dtype={"bf16": 0, "fp8": 1, "nvfp4": 2}[spec.kv_dtype])
    qsl = np.concatenate([[0], np.cumsum(spec.q_lens)]).astype(np.int32)
    items, parts = pkv.plan(cfg, qsl, np.asarray(spec.seq_lens, np.int32), num_sms)
    return items, parts, qsl


PF_PART_SLOTS = 32     # a split prefill item's partial: 256 rows = 32 decode slots


def _check_plan(spec, num_sms=152):
    items, parts, qsl = _plan(spec, num_sms)
    G = spec.hq // spec.hkv
    dec_keys = {}
    rows = {}
    ranges = {}
    slots = []
    for w in items:
        i, h = w["seq"], w["kv_head"]
        q, L = spec.q_lens[i], spec.seq_lens[i]
        assert w["tok0"] == qsl[i] and w["hist"] == L - q
        if w["kind"] == 0 and q * G <= 8:
            assert w["row0"] == 0 and w["n_rows"] == q * G
            dec_keys.setdefault((i, h), []).append((w["k_begin"], w["k_end"], w))
            if w["part"] >= 0:
                slots.append(w["part"])
        else:
            assert q * G > 8
            # G <= 128 uses tensor-core tiles (every pool format), larger
            # groups 8-row chunks on the decode kernel
            assert w["kind"] == (1 if G <= 128 else 0)
            if w["kind"] == 0:
                assert w["n_rows"] <= 8 and w["row0"] % 8 == 0 and w["part"] == -1
                assert w["k_begin"] == 0
            ranges.setdefault((i, h, w["row0"], w["n_rows"]), []).append(w)
            if w["k_begin"] == 0:
                rows.setdefault((i, h), []).append((w["row0"], w["n_rows"]))
            if w["part"] >= 0:
                slots.extend(range(w["part"], w["part"] + PF_PART_SLOTS))
    # decode: the ranges of each (request, KV head) tile [0, L) in order
    for (i, h), rs in dec_keys.items():
        rs.sort()
        assert rs[0][0] == 0 and rs[-1][1] == spec.seq_lens[i]
        for (a0, b0, _), (a1, b1, _) in zip(rs, rs[1:]):
            assert b0 == a1 and a1 % 256 == 0
        ns = len(rs)
        for k, (_, _, w) in enumerate(rs):
            assert w["n_split"] == ns
            if ns == 1:
                assert w["part"] == -1 and w["pair"] == -1
            else:
                assert w["part"] == w["pair"] + k          # contiguous slots
    # prefill: the key ranges of each row tile cover its causal reach in
    # order, split at multiples of 128 no later than the tile's first query
    # position (every row sees a key of every range)
    for (i, h, row0, n_rows), ws in ranges.items():
        ws.sort(key=lambda w: w["k_begin"])
        hist = spec.seq_lens[i] - spec.q_lens[i]
        reach = hist + (row0 + n_rows - 1) // G + 1
        assert ws[0]["k_begin"] == 0 and ws[-1]["k_end"] == reach
        ns = len(ws)
        for k, w in enumerate(ws):
            assert w["n_split"] == ns
            assert w["k_begin"] % max(128, spec.block_size) == 0
            assert w["k_begin"] <= hist + row0 // G
            if k + 1 < ns:
                assert w["k_end"] == ws[k + 1]["k_begin"]
            if ns == 1:
                assert w["part"] == -1 and w["pair"] == -1
            else:
                assert w["part"] == w["pair"] + PF_PART_SLOTS * k
    # prefill: tiles of each (request, KV head) cover rows [0, q*G)
    for (i, h), rs in rows.items():
        rs.sort()
        assert rs[0][0] == 0
        assert sum(n for _, n in rs) == spec.q_lens[i] * G
    assert sorted(slots) == list(range(parts))
    # the merge kernels take their groups from the head of each kind's list:
    # the first range of every split pair (decode) or row tile (prefill)
    # comes before any other item of that kind
    for kind in (0, 1):
        ws = [w for w in items if w["kind"] == kind]
        lead = [w["part"] >= 0 and w["part"] == w["pair"] for w in ws]
        n_lead = sum(lead)
        assert all(lead[:n_lead]) and not any(lead[n_lead:])
    # every (request, KV head) pair with tokens appears
    seen = set(dec_keys) | set(rows)
    assert len(seen) == sum(1 for q in spec.q_lens if q > 0) * spec.hkv
    return items, parts


@pytest.mark.parametrize("index", range(5))
def test_plan_covers_the_workloads(index):
    items, _ = _check_plan(workloads.config_spec(index))
    if index in (2, 3):
        # thousands of prefill tiles fill the machine: no key-range splits
        assert all(w["part"] == -1 for w in items if w["kind"] == 1)


@pytest.mark.parametrize("hq,hkv,q_lens,seq_lens", [
    (32, 8, [16], [32784]),                  # a few new tokens over a long history
    (32, 8, [64], [4160]),
    (8, 2, [64], [1064]),                    # the tiny prefill workload's shape
    (24, 8, [300], [2300]),                  # G = 3: rows in whole tokens
    (40, 8, [5, 77], [9000, 20077]),         # G = 5
    (32, 8, [1] * 6 + [48], [5000] * 6 + [40048]),   # decodes beside a small prefill
    (32, 8, [20], [100]),                    # short history: too few tiles to split
])
def test_small_prefills_split_their_key_ranges(hq, hkv, q_lens, seq_lens):
    spec = workloads.custom_spec("split", hq, hkv, 16, q_lens, seq_lens)
    items, parts = _check_plan(spec)
    pre = [w for w in items if w["kind"] == 1]
    tiles = sum((w["k_end"] - w["k_begin"] + 127) // 128 for w in pre)
    if max(seq_lens) >= 4096:
        # split: about one range per SM, each of at least two 128-key tiles
        assert any(w["n_split"] > 1 for w in pre)
        assert len(pre) <= 2 * 152 and parts <= 16384
        assert all((w["k_end"] - w["k_begin"] + 127) // 128 >= 1 for w in pre)
        assert max((w["k_end"] - w["k_begin"] + 127) // 128 for w in pre) <= \
            max(2, -(-2 * tiles // 152))
    if max(seq_lens) <= 128:
        assert all(w["n_split"] == 1 for w in pre)


def test_plan_orders_longest_first():
    items, _, _ = _plan(workloads.config_spec(3))
    dec = [w["k_end"] - w["k_begin"] for w in items if w["kind"] == 0]
    assert dec == sorted(dec, reverse=True)
    # prefill tiles: grouped by (request, KV head), groups longest first,
    # tiles longest first within a group
    pre = [w for w in items if w["kind"] == 1]
    groups = []
    for w in pre:
        key = (w["seq"], w["kv_head"])
        if not groups or groups[-1][0] != key:
            groups.append((key, []))
        groups[-1][1].append(w["k_end"] * w["n_rows"])
    assert len({g[0] for g in groups}) == len(groups)      # contiguous groups
    totals = [sum(c) for _, c in groups]
    assert totals == sorted(totals, reverse=True)
    for _, c in groups:
        assert c == sorted(c, reverse=True)


def test_plan_splits_fill_the_machine():
    items, parts, _ = _plan(workloads.config_spec(1))
    assert len(items) >= 4 * 152
    items, parts, _ = _plan(workloads.config_spec(4))
    assert len(items) >= 4 * 152 and parts <= 16384


def test_one_long_request_splits_into_many_ranges():
    """A lone 600K-token decode is cut into more than 32 ranges per (request,
    KV head) pair (the case the wide merge kernel serves), every range a
    multiple of 256 keys long except the last."""
    spec = workloads.custom_spec("long_one", 32, 8, 16, [1], [600_000])
    _check_plan(spec)
    items, parts, _ = _plan(spec)
    assert all(w["n_split"] > 32 for w in items)
    assert parts == len(items)


@pytest.mark.parametrize("qsl,lens,msg", [
    ([1, 2], [5], "query_start_loc_host[0]"),
    ([0, 3, 2], [5, 5], "decreases"),
    ([0, 6], [5], "less than"),
])
def test_plan_rejects_bad_metadata(qsl, lens, msg):
    cfg = pkv.make_config(8, 2, 16, 100, 4, 64)
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan(cfg, np.asarray(qsl, np.int32), np.asarray(lens, np.int32))
    assert e.value.status == 1 and msg in str(e.value)


def test_plan_empty_and_zero_token_requests():
    cfg = pkv.make_config(8, 2, 16, 100, 4, 64)
    items, parts = pkv.plan(cfg, np.asarray([0, 0, 3], np.int32), np.asarray([7, 9], np.int32))
    assert all(w["seq"] == 1 for w in items) and parts == 0
    items, parts = pkv.plan(cfg, np.asarray([0], np.int32), np.asarray([], np.int32))
    assert items == []


@pytest.mark.parametrize("kv,hq,hkv", [("nvfp4", 256, 1), ("bf16", 256, 1), ("fp8", 512, 2)])
def test_prefill_rows_without_tensor_core_tiles_are_chunked(kv, hq, hkv):
    """With query groups above 128, prefill rows become
    decode-kernel items of at most 8 rows: they tile [0, q*G) exactly, each
    reaches keys up to its last token's position, writes the output directly,
    and the chunks of one (request, KV head) are adjacent in launch order."""
    spec = workloads.custom_spec("chunks", hq, hkv, 16, [1, 40, 3, 130],
                                 [17, 300, 2000, 130], seed=3, kv_dtype=kv)
    items, parts, qsl = _plan(spec)
    G = hq // hkv
    assert all(w["kind"] == 0 for w in items)
    rows = {}
    order = []
    for w in items:
        i, h = w["seq"], w["kv_head"]
        q, L = spec.q_lens[i], spec.seq_lens[i]
        if q * G <= 8:
            continue
        assert w["k_begin"] == 0 and w["part"] == -1 and w["n_split"] == 1
        assert w["k_end"] == L - q + (w["row0"] + w["n_rows"] - 1) // G + 1
        rows.setdefault((i, h), []).append((w["row0"], w["n_rows"]))
        if not order or order[-1] != (i, h):
            order.append((i, h))
    assert len(order) == len(set(order))                   # contiguous groups
    for (i, h), rs in rows.items():
        rs.sort()
        assert [r0 for r0, _ in rs] == list(range(0, spec.q_lens[i] * G, 8))
        assert sum(n for _, n in rs) == spec.q_lens[i] * G
    chunked = {i for i, q in enumerate(spec.q_lens) if q * G > 8}
    assert set(rows) == {(i, h) for i in chunked for h in range(hkv)}
