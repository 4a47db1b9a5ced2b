"""Benchmark of the paged-KV attention hot path on one or more GB300s.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the hot path over the decode-batch workload (64
requests x 1 query token, contexts uniform in [4096, 32768], 32q/8kv heads,
head_dim 128, block_size 16, bf16 KV in a shuffled block pool): host plan,
KV append of the 64 new tokens (pkv_write_slots), split-KV decode with the
log-sum-exp combine (pkv_attention_varlen).  `value` is algorithmic bytes
(every context token's K and V once, Q and O, the append's read + write) per
second over the whole step, all inputs resident in HBM.  Each rank of a
multi-GPU run (torchrun) processes its own replica (weak scaling).  The
incremental-prefill (bf16, E4M3 and NVFP4 KV), mixed-step, FP8 and NVFP4 decode
workloads are reported in `secondary` unless --primary-only is given.

`--impl reference` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (one (request, KV head) slice per step).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode attn HBM GB/s (% of 8 TB/s); incr-prefill attn TFLOP/s (% bf16 peak)"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--primary-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None, choices=sorted(CASES),
                    help="time a reduced workload only (for profiler captures)")
    ap.add_argument("--no-stage", action="store_true",
                    help="with --case: no K/V staging pools (E4M3 / NVFP4 prefill "
                         "converts the codes inside the prefill kernel)")
    return ap.parse_args()


# Reduced workloads for profiler captures: the same kernels and shapes on a
# few of a workload's requests, still far larger than L2.
CASES = {
    "small-decode": (1, list(range(16))),     # ~1.3 GB of bf16 KV
    "small-prefill": (2, [4, 5]),             # two post-tool-call sessions
    "small-fp8": (4, [0]),                    # one ~0.6-1M-token FP8 request
    "small-nvfp4": (4, [0, 1]),               # two such requests, NVFP4 KV
    "small-prefill-fp8": (2, [4, 5]),         # two post-tool-call sessions, E4M3 KV
    "small-prefill-nvfp4": (2, [4, 5]),       # the same with NVFP4 KV
    "small-mixed": (3, [0, 40, 80, 119, 127]),   # 4 decodes + the 392-token chunk, ~2 GB
    # the whole post-tool-call step, for captures of its 26K-token KV append
    # (216 MB bf16, 162 MB E4M3, 138 MB NVFP4 per launch)
    "append-c3": (2, list(range(16))),
    "append-c3-fp8": (2, list(range(16))),
    "append-c3-nvfp4": (2, list(range(16))),
}
CASE_KV = {"small-nvfp4": "nvfp4", "small-prefill-fp8": "fp8", "small-prefill-nvfp4": "nvfp4",
           "append-c3-fp8": "fp8", "append-c3-nvfp4": "nvfp4"}


def case_spec(name: str) -> W.Spec:
    index, seqs = CASES[name]
    full = W.config_spec(index)
    kv = CASE_KV.get(name, full.kv_dtype)
    whole = seqs == list(range(full.num_seqs))
    return W.Spec(f"{full.name}[{name}]", full.hq, full.hkv, full.block_size,
                  kv, [full.q_lens[i] for i in seqs],
                  [full.seq_lens[i] for i in seqs], full.seed,
                  shared_prefix=full.shared_prefix if whole else None)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK)
    d["source"] = "fallback"
    return d


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        samples = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                samples.append((ts, float(f[2]), float(f[3]), f[5:9]))
            except (ValueError, IndexError):
                continue
        inside = [s for s in samples if t0 - 0.15 <= s[0] <= t1 + 0.15] or samples
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3])
                          if v.lower() == "active"})
        return {"sm_mhz": float(np.median([s[1] for s in inside])),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside)}


def traffic_from_profile(summary: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel's
    sources are unchanged since: the summary lists them (`sources:`) and the
    sha256 of their concatenation (`source_sha256:`)."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"^sources:\s*(.+)$", text, re.M)
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"traffic_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_sha or not m_tr:
        return None
    return float(m_tr.group(1)) if sources_sha256(m_src.group(1).split()) == m_sha.group(1) \
        else None


def sources_sha256(names) -> str | None:
    h = hashlib.sha256()
    for n in names:
        f = os.path.join(ROOT, "paged_kv_attention_pkv_gb300", "csrc", n)
        if not os.path.exists(f):
            return None
        h.update(open(f, "rb").read())
    return h.hexdigest()


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- our arm --

def make_handle(batch, flags, stage=True):
    """A handle for the step; E4M3 / NVFP4 pools get K/V staging pools with
    room for every request's context (the staged tensor-core prefill) unless
    stage=False."""
    import paged_kv_attention_pkv_gb300 as pkv
    s = batch.spec
    stage_tokens = (sum(W.cdiv(L, s.block_size) * s.block_size for L in s.seq_lens)
                    if stage and s.kv_dtype != "bf16" else 0)
    cfg = pkv.make_config(s.hq, s.hkv, s.block_size, batch.num_blocks, s.num_seqs,
                          s.num_tokens, softmax_scale=s.softmax_scale, flags=flags,
                          kv_dtype={"bf16": pkv.KV_BF16, "fp8": pkv.KV_FP8_E4M3,
                                    "nvfp4": pkv.KV_NVFP4}[s.kv_dtype],
                          stage_tokens=stage_tokens)
    return pkv.Handle(cfg, device=batch.q.device.index or 0)


def device_meta(batch):
    dev = batch.q.device
    return {"slots": torch.from_numpy(batch.slot_mapping).to(dev),
            "qsl": torch.from_numpy(batch.qsl).to(dev),
            "lens": torch.from_numpy(batch.seq_lens).to(dev),
            "bt": torch.from_numpy(batch.block_tables).to(dev)}


def time_workload(index, steps: int, warmup: int, world: int, peaks: dict,
                  device: str, sampler: ClockSampler | None = None, e2e: bool = False,
                  separate: bool = False, stage: bool = True):
    import paged_kv_attention_pkv_gb300 as pkv

    spec = W.config_spec(index) if isinstance(index, int) else index
    batch = W.generate(spec, device)
    work = W.algorithmic_work(spec)
    h = make_handle(batch, pkv.FLAG_TIMING | (pkv.FLAG_SEPARATE if separate else 0), stage)
    m = device_meta(batch)
    out = torch.empty_like(batch.q)
    stream = torch.cuda.current_stream()

    def step():
        h.write_slots(batch.k_new, batch.v_new, m["slots"], batch.k_cache,
                      batch.v_cache, batch.k_scale, batch.v_scale, stream=stream)
        h.attention_varlen(batch.q, batch.k_cache, batch.v_cache, m["qsl"], m["lens"],
                           m["bt"], batch.qsl, batch.seq_lens, out=out,
                           k_scale=batch.k_scale, v_scale=batch.v_scale, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    h.timing_reset()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    w0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    if sampler:
        time.sleep(0.2)
        sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    per_kind = {}
    for kind, name in ((pkv.KERNEL_APPEND, "append"), (pkv.KERNEL_DECODE, "decode"),
                       (pkv.KERNEL_PREFILL, "prefill"), (pkv.KERNEL_MIXED, "mixed"),
                       (pkv.KERNEL_MERGE, "merge"), (pkv.KERNEL_STAGE, "stage")):
        n, tot = h.timing_read(kind)
        if n:
            per_kind[name] = (n, tot / n)
    # every step launches each kind it uses once (the timing ring keeps the
    # first 4096 launches of each kind)
    assert all(n == min(steps, 4096) for n, _ in per_kind.values()), per_kind
    launches_per_step = len(per_kind)
    res = {"spec": spec, "work": work, "ms": ms, "steps": steps, "kinds": per_kind,
           "gpu_launches": launches_per_step * steps, "wall": (w0, w1)}
    if e2e:
        res["e2e"] = time_e2e(h, batch, m, out, min(steps, 300), stream, world)
    h.close()
    del batch
    torch.cuda.empty_cache()
    return res


def time_e2e(h, batch, m, out, steps, stream, world):
    """Same step through the public API with the step's inputs in pinned host
    memory: H2D of q, new K/V, slots and metadata, the step, D2H of out.
    Copies run on two copy streams, double-buffered as a serving loop would
    run them: step i+1's inputs go up while step i computes, step i's output
    comes back while step i+1 computes.  The timed region opens before the
    first upload and closes after the last download."""
    src = {"q": batch.q, "k_new": batch.k_new, "v_new": batch.v_new, "slots": m["slots"],
           "qsl": m["qsl"], "lens": m["lens"], "bt": m["bt"]}
    # the step's inputs packed into one pinned buffer (256-byte aligned
    # fields), brought over with one copy into one of two device buffers
    offs, total = {}, 0
    for k, v in src.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=batch.q.device) for _ in range(2)]
    devs = [{}, {}]
    for k, v in src.items():
        n = v.numel() * v.element_size()
        host_buf[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8).cpu())
        for b in range(2):
            devs[b][k] = dev_bufs[b][offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
    outs = [out, torch.empty_like(out)]
    out_hosts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in src.values())
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()   # noqa: E731
    uploaded = [ev(), ev()]     # inputs of buffer b are on the device
    consumed = [ev(), ev()]     # the step reading buffer b (and writing out b) is done
    fetched = [ev(), ev()]      # out b is back on the host

    def upload(i):
        b = i & 1
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(consumed[b])
            dev_bufs[b].copy_(host_buf, non_blocking=True)
            uploaded[b].record(up)

    def run(n):
        upload(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(uploaded[b])
            if i >= 2:
                stream.wait_event(fetched[b])
            d = devs[b]
            h.write_slots(d["k_new"], d["v_new"], d["slots"], batch.k_cache,
                          batch.v_cache, batch.k_scale, batch.v_scale, stream=stream)
            h.attention_varlen(d["q"], batch.k_cache, batch.v_cache, d["qsl"], d["lens"],
                               d["bt"], batch.qsl, batch.seq_lens, out=outs[b],
                               k_scale=batch.k_scale, v_scale=batch.v_scale, stream=stream)
            consumed[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(consumed[b])
                out_hosts[b].copy_(outs[b], non_blocking=True)
                fetched[b].record(down)
        for b in range(min(n, 2)):
            stream.wait_event(fetched[b])

    run(3)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_stream(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    return {"ms_per_step": ms / steps, "h2d": h2d, "d2h": d2h, "steps": steps,
            "copies": "two copy streams, double-buffered (uploads of step i+1 and the "
                      "download of step i overlap step i+1's kernels)"}


def roofline_decode(res, peaks, traffic):
    n, avg_ms = res["kinds"]["decode"]
    byts = res["work"]["decode_bytes"]
    ach = byts / (avg_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": "decode_kernel<bf16>", "achieved": round(ach, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4),
            "peak_source": f"{peaks['source']} (hbm_gbs)",
            "avg_launch_ms": round(avg_ms, 5), "launches": n,
            "algorithmic_bytes_per_launch": byts, "traffic": traffic}


def cpu_baseline(min_seconds: float = 10.0):
    """The oracle, as it stands, on the decode batch: whole passes (all 64
    requests, all heads, its own append + attention) repeated until at least
    `min_seconds` of CPU time have been spent."""
    import oracle

    from tests import gpu_util as U
    spec = W.config_spec(1)
    batch = W.generate(spec, "cuda")
    sub = W.subset(batch, list(range(spec.num_seqs)))
    del batch
    torch.cuda.empty_cache()
    passes = 0
    t0 = time.perf_counter()
    while True:
        U.oracle_subset(sub, spec)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= 50:
            break
    byts = passes * sum(int(L) * 2 * spec.hkv * 128 * 2 for L in spec.seq_lens)
    return {"value": round(byts / dt / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{passes} whole passes over the decode batch (64 requests, 32 heads, "
                      f"append + attention, fp64), {dt:.1f} s",
            "seconds": round(dt, 2)}


def run_case(args, local_rank):
    peaks = load_peaks()
    r = time_workload(case_spec(args.case), args.steps, args.warmup, 1, peaks,
                      f"cuda:{local_rank}", stage=not args.no_stage)
    work = r["work"]
    ent = {"case": r["spec"].name, "ms_per_step": r["ms"] / args.steps,
           "kernel_ms": {k: v[1] for k, v in r["kinds"].items()}, "work": work}
    print(json.dumps(ent), flush=True)


def run_ours(args, rank, world, local_rank):
    import paged_kv_attention_pkv_gb300 as pkv
    pkv.load()
    torch.cuda.set_device(local_rank)
    device = f"cuda:{local_rank}"
    if args.case:
        return run_case(args, local_rank)
    peaks = load_peaks()
    sampler = ClockSampler(local_rank) if rank == 0 or world > 1 else None
    prim = time_workload(1, args.steps, args.warmup, world, peaks, device,
                         sampler=sampler, e2e=True)
    spec, work = prim["spec"], prim["work"]
    bytes_step = work["decode_bytes"] + work["append_bytes"]
    ms_step = prim["ms"] / args.steps
    value = world * bytes_step / (ms_step * 1e-3) / 1e9
    e2e = prim["e2e"]
    e2e_value = world * bytes_step / (e2e["ms_per_step"] * 1e-3) / 1e9
    traffic = traffic_from_profile("ncu_decode_c2.md")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; shapes of the decode-batch workload)",
        "config": {"workload": spec.name, "requests": spec.num_seqs,
                   "context": "uniform [4096, 32768]", "q_heads": spec.hq,
                   "kv_heads": spec.hkv, "head_dim": 128, "block_size": spec.block_size,
                   "kv_bytes": work["decode_bytes"], "append_tokens": spec.num_tokens,
                   "l2": "no flush: 5.1 GB of KV per step, far above the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline_decode(prim, peaks, traffic),
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e["ms_per_step"], 5)},
        "gpu_launches": prim["gpu_launches"],
        "clocks": sampler.summary(*prim["wall"]) if sampler else None,
        "kernel_ms": {k: round(v[1], 5) for k, v in prim["kinds"].items()},
    }
    if not args.primary_only:
        line["secondary"] = secondary(args, world, peaks, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_graph(index, steps: int, device: str) -> dict:
    """One step (append + attention) of a workload issued eagerly `steps`
    times back to back, against the same step captured once in a CUDA graph
    and replayed `steps` times; CUDA events around each whole loop, so host
    enqueue time shows wherever it exceeds the GPU time."""
    import paged_kv_attention_pkv_gb300 as pkv
    spec = W.config_spec(index)
    batch = W.generate(spec, device)
    h = make_handle(batch, 0)
    m = device_meta(batch)
    out = torch.empty_like(batch.q)
    stream = torch.cuda.current_stream()

    def step():
        h.write_slots(batch.k_new, batch.v_new, m["slots"], batch.k_cache,
                      batch.v_cache, batch.k_scale, batch.v_scale)
        h.attention_varlen(batch.q, batch.k_cache, batch.v_cache, m["qsl"], m["lens"],
                           m["bt"], batch.qsl, batch.seq_lens, out=out,
                           k_scale=batch.k_scale, v_scale=batch.v_scale)

    def loop(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    eager_ms = loop(step)
    h.graph_prepare(batch.qsl, batch.seq_lens)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    graph_ms = loop(g.replay)
    h.close()
    del g, batch
    torch.cuda.empty_cache()
    return {"workload": spec.name, "steps": steps, "eager_ms_per_step": round(eager_ms, 5),
            "graph_ms_per_step": round(graph_ms, 5), "speedup": round(eager_ms / graph_ms, 3)}


def time_per_call(index, device: str, calls: int = 20, warmup: int = 5) -> dict:
    """Latency of single steps (append + attention): `warmup` untimed calls,
    then `calls` calls each bracketed by CUDA events with the device idle
    before it, so a call's span includes its host-side enqueue.  "warm" runs
    the calls back to back; "cold" writes a 256 MB buffer (twice the L2)
    before each call, outside its events.  The library's own per-kernel
    events give the device time of the kernels alone."""
    import paged_kv_attention_pkv_gb300 as pkv
    spec = W.config_spec(index) if isinstance(index, int) else index
    batch = W.generate(spec, device)
    h = make_handle(batch, pkv.FLAG_TIMING)
    m = device_meta(batch)
    out = torch.empty_like(batch.q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def step():
        h.write_slots(batch.k_new, batch.v_new, m["slots"], batch.k_cache,
                      batch.v_cache, batch.k_scale, batch.v_scale)
        h.attention_varlen(batch.q, batch.k_cache, batch.v_cache, m["qsl"], m["lens"],
                           m["bt"], batch.qsl, batch.seq_lens, out=out,
                           k_scale=batch.k_scale, v_scale=batch.v_scale)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    res = {"workload": spec.name, "calls": calls, "warmup": warmup}
    for mode in ("warm", "cold"):
        h.timing_reset()
        spans = []
        for i in range(calls):
            if mode == "cold":
                flush.fill_(i & 0xFF)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            step()
            e1.record()
            torch.cuda.synchronize()
            spans.append(e0.elapsed_time(e1) * 1e3)
        kernels_us = 0.0
        for kind in (pkv.KERNEL_APPEND, pkv.KERNEL_DECODE, pkv.KERNEL_PREFILL,
                     pkv.KERNEL_MIXED, pkv.KERNEL_MERGE, pkv.KERNEL_STAGE):
            n, tot = h.timing_read(kind)
            if n:
                kernels_us += tot / n * 1e3
        res[mode] = {"median_us": round(float(np.median(spans)), 2),
                     "min_us": round(float(np.min(spans)), 2),
                     "kernels_mean_us": round(kernels_us, 2)}
    h.close()
    del batch, flush
    torch.cuda.empty_cache()
    return res


def secondary(args, world, peaks, device):
    out = []
    # one session's post-tool-call prefill alone: 64 new tokens over a
    # 48000-token history (the median of the post-tool-call workload)
    one_session = W.custom_spec("one_session_post_tool_prefill_q64_h48000", 32, 8, 16,
                                [64], [48064], seed=1002)
    out.append({"per_call": [time_per_call(0, device), time_per_call(1, device),
                             time_per_call(one_session, device)]})
    out.append({"cuda_graph": [time_graph(0, 500, device), time_graph(1, 200, device)]})
    nvfp4 = dataclasses.replace(W.config_spec(4), name="c5_nvfp4_long_decode",
                                kv_dtype="nvfp4")
    fp8_pf = dataclasses.replace(W.config_spec(2), name="c3_fp8_post_tool_prefill",
                                 kv_dtype="fp8")
    nv_pf = dataclasses.replace(W.config_spec(2), name="c3_nvfp4_post_tool_prefill",
                                kv_dtype="nvfp4")
    gpu_index = int(device.split(":")[1]) if ":" in device else 0
    for idx, steps in ((2, 10), (fp8_pf, 10), (nv_pf, 5), (3, 10), (4, 50), (nvfp4, 50)):
        # clocks sampled during each timed loop: the tensor-bound steps run
        # at the power cap's clocks once the GPU is warm
        smp = ClockSampler(gpu_index)
        r = time_workload(idx, steps, 3, world, peaks, device, sampler=smp)
        spec, work = r["spec"], r["work"]
        unstaged = None
        if "stage" in r["kinds"]:
            # the same step with no staging pools: the prefill kernel converts
            # the E4M3 / NVFP4 codes itself
            u = time_workload(idx, steps, 3, world, peaks, device, stage=False)
            n, avg = u["kinds"]["prefill"]
            tf = work["prefill_flops"] / (avg * 1e-3) / 1e12
            unstaged = {"ms_per_step": round(u["ms"] / steps, 4),
                        "kernel_ms": {k: round(v[1], 4) for k, v in u["kinds"].items()},
                        "prefill": {"value": round(tf, 1), "unit": "TFLOP/s",
                                    "frac": round(tf / peaks["bf16_tflops"], 4)}}
        ms_step = r["ms"] / steps
        ent = {"workload": spec.name, "ms_per_step": round(ms_step, 4),
               "kernel_ms": {k: round(v[1], 4) for k, v in r["kinds"].items()},
               "clocks": smp.summary(*r["wall"])}
        if "mixed" in r["kinds"]:
            # one launch for both kinds; the per-kind figures below come from
            # the same step run as separate decode and prefill launches
            n, avg = r["kinds"]["mixed"]
            t_ideal = (work["decode_bytes"] / (peaks["hbm_gbs"] * 1e9) +
                       work["prefill_flops"] / (peaks["bf16_tflops"] * 1e12))
            ent["mixed"] = {"kernel_ms": round(avg, 4),
                            "roofline_frac": round(t_ideal / (avg * 1e-3), 4),
                            "note": "ideal time (decode bytes at HBM peak + prefill "
                                    "flops at bf16 peak) / mixed-launch time"}
            r = time_workload(idx, steps, 3, world, peaks, device, separate=True)
            ent["separate"] = {"ms_per_step": round(r["ms"] / steps, 4),
                               "kernel_ms": {k: round(v[1], 4)
                                             for k, v in r["kinds"].items()}}
        if work["prefill_flops"]:
            n, avg = r["kinds"]["prefill"]
            # E4M3 / NVFP4 KV: the K/V staging kernel counts as prefill time
            avg += r["kinds"].get("stage", (0, 0.0))[1]
            tf = work["prefill_flops"] / (avg * 1e-3) / 1e12
            peak = peaks["bf16_tflops"]
            # staged E4M3 / NVFP4 KV runs the bf16 kernel on bf16 K/V; unstaged,
            # E4M3 KV runs QK as two FP8 MMAs (query hi + lo parts) and PV in
            # f16, NVFP4 KV both in f16: the tensor time of the bf16 kernel
            # either way, so the same bf16 peak applies
            ent["prefill"] = {"value": round(tf, 1), "unit": "TFLOP/s", "bound": "tensor",
                              "frac": round(tf / peak, 4), "peak": peak,
                              "peak_source": f"{peaks['source']} (bf16_tflops)",
                              "flops_per_launch": work["prefill_flops"],
                              "ms": round(avg, 4),
                              "includes": "K/V staging + prefill" if "stage" in r["kinds"]
                              else "prefill"}
            if unstaged:
                ent["unstaged"] = unstaged
        if work["decode_bytes"]:
            n, avg = r["kinds"]["decode"]
            # the decode kernel and the merge of its split ranges
            avg += r["kinds"].get("merge", (0, 0.0))[1]
            gb = work["decode_bytes"] / (avg * 1e-3) / 1e9
            ent["decode"] = {"value": round(gb, 1), "unit": "GB/s", "bound": "hbm",
                             "frac": round(gb / peaks["hbm_gbs"], 4),
                             "peak": peaks["hbm_gbs"],
                             "bytes_per_launch": work["decode_bytes"],
                             "ms": round(avg, 4), "includes": "decode kernel + range merge"}
        if work["prefill_flops"] and work["decode_bytes"]:
            t_ideal = (work["decode_bytes"] / (peaks["hbm_gbs"] * 1e9) +
                       work["prefill_flops"] / (peaks["bf16_tflops"] * 1e12))
            ent["combined_roofline_frac"] = round(t_ideal / (ms_step * 1e-3), 4)
        n, avg = r["kinds"]["append"]
        ent["append"] = {"value": round(work["append_bytes"] / (avg * 1e-3) / 1e9, 1),
                         "unit": "GB/s", "bytes_per_launch": work["append_bytes"]}
        out.append(ent)
    return out


# ---------------------------------------------------------- reference arm --

def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, one (request, KV head) slice of the
    decode batch per step (its 4 query heads over the whole context)."""
    if rank != 0:
        return
    import oracle
    from tests import gpu_util as U
    full = W.config_spec(1)
    # one-KV-head slice of the workload: same lengths, same per-row work
    spec = W.Spec(full.name + "_kvslice", 4, 1, full.block_size, full.kv_dtype,
                  full.q_lens, full.seq_lens, full.seed)
    batch = W.generate(spec, "cpu")
    subs = [W.subset(batch, [i]) for i in range(spec.num_seqs)]
    del batch

    def step(i):
        s = subs[i % len(subs)]
        U.oracle_subset(s, spec)
        return int(s["seq_lens"][0]) * 2 * 128 * 2

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    byts = 0
    for i in range(args.steps):
        byts += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = byts / dt / 1e9
    cores = oracle.num_threads()
    sample = ("one (request, KV head) slice of the decode batch per step: 4 query "
              "heads over the request's whole context, fp64 oracle incl. its append")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes of the decode-batch workload)",
            "config": {"workload": full.name, "requests": full.num_seqs,
                       "context": "uniform [4096, 32768]", "q_heads": full.hq,
                       "kv_heads": full.hkv, "head_dim": 128,
                       "block_size": full.block_size, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
