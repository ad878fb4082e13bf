"""Benchmark of the MLA speculative-verify decode on GB300.

One step (default workload `sweep`) = one verify-decode call for each point of the
q x ctx sweep of sglang PR #33650 ("Raw q x ctx sweep" table) that fits the task's
configurations: H = 12, q in {1, 2, 4, 8} at ctx = 131072 with a bf16 paged cache, and
q = 8 at ctx = 1,048,576 with a bf16 cache and with an fp8 e4m3 cache. `value` is the
mean device time per call in microseconds over the step's calls; each call's KV
bandwidth and roofline fractions go beside it in `per_call`.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                        [--workload sweep|sweep131k|contig4096|long_bf16|long_fp8|h96|ragged48|ragged128|prefill]

Timing: each call is captured R times back to back (--graph-calls, default 4) in one
CUDA graph, every copy reading a cache of its own, and the graph replay is bracketed by
CUDA events on the stream it runs on; time per call = graph time / R. (A serving engine
replays the whole decode step as one graph, so this leaves out the per-graph launch gap
of a graph that holds a single call.) Every call reads a cache that no call since it
was last read has left in L2: the R copies of a call and the calls of a step together
are many times the 126 MB L2. With --l2 flush a 256 MB write before every graph replay
also evicts everything else.
SM clocks and throttle reasons are sampled with nvidia-smi during the timed region.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mla_speculative_verify_gb300 import inputs  # noqa: E402

METRIC = "MLA verify-decode µs/call and KV GB/s as % of GB300 HBM peak, q×ctx sweep"
L2_FLUSH_BYTES = 256 << 20
# GB300 HBM3e bandwidth as rated by the vendor (nominal; the measured copy peak of
# MEASURED_PEAKS.json is the roofline denominator, this one is reported beside it)
HBM_RATED_GBS = 7900.0
CSRC = os.path.join(ROOT, "mla_speculative_verify_gb300", "csrc")


def workload(name: str):
    """List of problems making up one step, and a description."""
    if name == "sweep":
        probs = [inputs.workload_sweep_131k(q) for q in (1, 2, 4, 8)]
        probs += [inputs.workload_long(inputs.KV_BF16), inputs.workload_long(inputs.KV_FP8)]
        return probs, dict(workload="h12_sweep_q1-2-4-8_ctx131072_bf16+q8_ctx1048576_bf16+fp8", H=12,
                           ctx=[131072, 1 << 20], q=[1, 2, 4, 8], kv=["bf16", "fp8_e4m3"], page_size=64)
    if name == "sweep131k":
        return [inputs.workload_sweep_131k(q) for q in (1, 2, 4, 8)], dict(
            workload="h12_ctx131072_bf16_q1-2-4-8", H=12, ctx=131072, q=[1, 2, 4, 8], kv="bf16", page_size=64)
    if name == "grid":
        # every cell of a q x ctx x cache-dtype sweep: q 1/2/4/8, ctx 131072 / 524288 / 1048576
        ctxs = (131072, 1 << 19, 1 << 20)
        probs = [inputs.workload_sweep_131k(q, ctx=c, kv_dtype=kv) for kv in (inputs.KV_BF16, inputs.KV_FP8)
                 for c in ctxs for q in (1, 2, 4, 8)]
        return probs, dict(workload="h12_q1-2-4-8_ctx131072-524288-1048576_bf16+fp8", H=12, ctx=list(ctxs),
                           q=[1, 2, 4, 8], kv=["bf16", "fp8_e4m3"], page_size=64)
    if name == "sweep131k_fp8":
        return [inputs.workload_sweep_131k(q, kv_dtype=inputs.KV_FP8) for q in (1, 2, 4, 8)], dict(
            workload="h12_ctx131072_fp8_q1-2-4-8", H=12, ctx=131072, q=[1, 2, 4, 8], kv="fp8_e4m3", page_size=64)
    if name == "contig4096":
        return [inputs.workload_contiguous_small()], dict(workload="h12_q2_ctx4096_bf16_contiguous", H=12, ctx=4096,
                                                         q=[2], kv="bf16", page_size=64)
    if name == "long_bf16":
        return [inputs.workload_long(inputs.KV_BF16)], dict(workload="h12_q8_ctx1048576_bf16", H=12, ctx=1 << 20, q=[8],
                                                             kv="bf16", page_size=64)
    if name == "long_bf16_q1":
        return [inputs.workload_long(inputs.KV_BF16, q=1)], dict(workload="h12_q1_ctx1048576_bf16", H=12,
                                                                  ctx=1 << 20, q=[1], kv="bf16", page_size=64)
    if name == "long_fp8":
        return [inputs.workload_long(inputs.KV_FP8)], dict(workload="h12_q8_ctx1048576_fp8", H=12, ctx=1 << 20, q=[8],
                                                            kv="fp8_e4m3", page_size=64)
    if name == "h96":
        probs = [inputs.workload_h96(q, c, kv) for q in (1, 8) for c in (32768, 131072) for kv in ("bf16", "fp8")]
        return probs, dict(workload="h96_q1-8_ctx32768-131072_bf16-fp8", H=96, page_size=64)
    if name == "prefill":
        probs = [inputs.make_problem(H, [131072], [2048], inputs.KV_BF16, seed=1006, name=f"h{H}_q2048_ctx131072_bf16")
                 for H in (12, 96)]
        return probs, dict(workload="prefill_h12+h96_q2048_ctx131072_bf16", H=[12, 96], q=2048, ctx=131072,
                           page_size=64)
    if name.startswith("ragged"):
        H = int(name[len("ragged"):])
        return [inputs.workload_ragged(H, "ragged"), inputs.workload_ragged(H, "uniform")], dict(
            workload=f"h{H}_b32_mtp3_ragged+uniform_q4_ctx16k-32k_fp8", H=H, page_size=64)
    raise SystemExit(f"unknown workload {name}")


def algorithmic_bytes(prob) -> int:
    """KV read once per request + Q + out + LSE + page table (bytes per call)."""
    kvb = 2 if prob.kv_dtype == inputs.KV_BF16 else 1
    H = prob.H
    tq = prob.total_q
    pages = int(((prob.seq_lens + 63) // 64).sum())
    return int(prob.seq_lens.astype(np.int64).sum()) * 576 * kvb + tq * H * 576 * 2 + tq * H * 512 * 2 + tq * H * 4 + pages * 4


def algorithmic_flops(prob) -> float:
    f = 0.0
    for ctx, q in zip(prob.seq_lens, prob.q_lens):
        vis = sum(int(ctx) - int(q) + i + 1 for i in range(int(q)))
        f += vis * prob.H * 2176.0
    return f


def kernel_source_hash() -> str:
    """sha256[:16] over the library's CUDA sources (sorted), recorded in each ncu summary.
    Comments and whitespace are left out (the sources hold no "//" or "/*" inside string
    literals), so a change to the code changes it and an edit of a comment does not."""
    import hashlib
    import re

    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(CSRC, name)).read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(name.encode())
            h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(profile_md: str) -> dict:
    """DRAM read + write bytes of one fold-kernel launch per call name, from a committed
    ncu summary (lines `traffic[<call>]: <bytes>`); empty when the summary is missing or
    the kernel sources changed since its counters were taken (it records their hash)."""
    import re

    try:
        text = open(profile_md).read()
    except OSError:
        return {}
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_sha or m_sha.group(1) != kernel_source_hash():
        return {}
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"traffic\[([\w.+-]+)\]:\s*(\d+)", text)}


def mma_dtype(prob) -> str:
    """Arithmetic type of a call's tensor-core products: bf16 x bf16 for a bf16 cache; for
    an e4m3 cache e4m3 x e4m3 on the stored codes and on two-part (hi + lo) e4m3 operands
    of Q and P; fp32 accumulation and softmax either way."""
    return "bf16" if prob.kv_dtype == inputs.KV_BF16 else "e4m3 (hi+lo operands)"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling (every 20 ms, each sample time-stamped) of the SM clock and the
    throttle reasons while the bench runs. The summary keeps the samples taken between
    `begin()` and `end()` (the timed region); when that region is shorter than three
    sampling periods it also keeps those of the warm-up just before it (same work), and
    says so."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import tempfile

        self.gpu = gpu_index
        self.proc = None
        self.t_warm = self.t_begin = self.t_end = None
        fd, self.path = tempfile.mkstemp(prefix=f"mla_bench_clocks_gpu{gpu_index}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def warmup(self):
        self.t_warm = time.time()

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    @staticmethod
    def parse(text: str):
        """(time in s since the epoch or None, fields after the time stamp) per sample line."""
        import datetime

        rows = []
        for line in text.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = None
            rows.append((t, parts[1:]))
        return rows

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        with open(self.path) as fh:
            text = fh.read()
        try:
            os.remove(self.path)
        except OSError:
            pass
        return self.summarize(self.parse(text), self.t_warm, self.t_begin, self.t_end)

    @staticmethod
    def summarize(rows, t_warm, t_begin, t_end):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = "whole run"
        if t_begin is not None and t_end is not None and all(t is not None for t, _ in rows):
            timed = [r for r in rows if t_begin <= r[0] <= t_end]
            window = "timed region"
            if len(timed) < 3 and t_warm is not None:
                timed = [r for r in rows if t_warm <= r[0] <= t_end]
                window = "warm-up + timed region"
            if timed:
                rows = timed
            else:
                window = "whole run (no sample in the timed region)"
        sm, smax, reasons = [], [], set()
        for _, parts in rows:
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        med = statistics.median(sm)
        return {"sm_mhz": med, "sm_max_mhz": max(smax), "reasons": sorted(reasons), "samples": len(sm),
                "window": window, "below_70pct_of_max": med < 0.7 * max(smax)}


def run_ours(args, probs, desc, rank, world):
    from mla_speculative_verify_gb300.decoder import VerifyDecoder

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    calls = []
    R = args.graph_calls
    for prob in probs:
        dec = VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype, dev)
        q = prob.q.to(dev)
        kv = prob.kv.to(dev)
        kvs = [kv] + [kv.clone() for _ in range(R - 1)]  # a cache of its own for every copy of the call
        pt = torch.from_numpy(prob.page_table).to(dev)
        out = torch.empty((prob.total_q, prob.H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((prob.total_q, prob.H), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            dec.run(q, kv, pt, out, lse, prob.sm_scale, prob.kv_scale, status)  # sets attributes, warms caches
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for r in range(R):
                    dec.run(q, kvs[r], pt, out, lse, prob.sm_scale, prob.kv_scale, status)
        calls.append(dict(prob=prob, dec=dec, q=q, kv=kv, kvs=kvs, pt=pt, out=out, lse=lse, status=status, graph=g))
    launches_per_step = R * sum(1 + (1 if c["dec"].info["n_merge"] > 0 else 0) for c in calls)

    def one_step(timed: bool):
        evs = []
        for c in calls:
            with torch.cuda.stream(stream):
                if args.l2 == "flush":
                    flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                c["graph"].replay()
                e1.record(stream)
            evs.append((e0, e1))
        return evs

    all_evs = []
    with ClockSampler(dev.index) as clk:
        clk.warmup()
        for _ in range(args.warmup):
            one_step(False)
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        clk.begin()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            all_evs.append(one_step(True))
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        clk.end()
    if world > 1:
        torch.distributed.barrier()
    graph_ms = np.array([[e0.elapsed_time(e1) for (e0, e1) in evs] for evs in all_evs])  # [K, calls]
    step_ms = graph_ms.sum(1)  # a step replays every call's graph: R calls of each
    per_call_ms = graph_ms / R
    status_bits = 0
    for c in calls:
        status_bits |= int(c["status"].item())
    # end to end: host (pinned) inputs copied in and the result read back inside the timed region
    if world > 1:
        torch.distributed.barrier()
    e2e = measure_e2e(args, calls, dev, stream)
    return dict(per_call_ms=per_call_ms, step_ms=step_ms, wall=wall, clocks=clk.summary(), status=status_bits,
                launches=launches_per_step * args.steps, e2e=e2e, calls=calls)


def measure_e2e(args, calls, dev, stream):
    """Same metric through the public API with host buffers: per call the H2D copy of
    q, the cache, the page table and the lengths, the decode, and the D2H of out and lse.
    The H2D copies run on a copy stream and each call's decode waits for its own inputs,
    so a call's decode (and its D2H, the other direction of the link) overlaps the next
    call's copies, as a serving loop would arrange it. Pinned-memory H2D tops out near
    210 GB/s on the GB300 machine whatever the number of streams, so the copies set the pace."""
    hosts = []
    for c in calls:
        prob = c["prob"]
        h = dict(q=prob.q.pin_memory(), kv=prob.kv.pin_memory(), pt=torch.from_numpy(prob.page_table).pin_memory(),
                 sl=torch.from_numpy(prob.seq_lens).pin_memory(), ql=torch.from_numpy(prob.q_lens).pin_memory(),
                 out=torch.empty(c["out"].shape, dtype=torch.bfloat16).pin_memory(),
                 lse=torch.empty(c["lse"].shape, dtype=torch.float32).pin_memory())
        hosts.append(h)
    h2d = sum(h["q"].numel() * 2 + h["kv"].numel() * h["kv"].element_size() + h["pt"].numel() * 4 +
              h["sl"].numel() * 8 for h in hosts)
    d2h = sum(h["out"].numel() * 2 + h["lse"].numel() * 4 for h in hosts)
    steps = max(1, min(args.steps, 5))
    copy_stream = torch.cuda.Stream(dev)

    def step():
        ready = []
        for c, h in zip(calls, hosts):
            with torch.cuda.stream(copy_stream):
                c["q"].copy_(h["q"], non_blocking=True)
                c["kv"].copy_(h["kv"], non_blocking=True)
                c["pt"].copy_(h["pt"], non_blocking=True)
                c["dec"].seq_lens_dev.copy_(h["sl"], non_blocking=True)
                c["dec"].q_lens_dev.copy_(h["ql"], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                ready.append(ev)
        for c, h, ev in zip(calls, hosts, ready):
            stream.wait_event(ev)
            with torch.cuda.stream(stream):
                c["dec"].run(c["q"], c["kv"], c["pt"], c["out"], c["lse"], c["prob"].sm_scale, c["prob"].kv_scale,
                             c["status"], stream=stream)
                h["out"].copy_(c["out"], non_blocking=True)
                h["lse"].copy_(c["lse"], non_blocking=True)
        copy_stream.synchronize()
        stream.synchronize()

    step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(copy_stream)
    stream.wait_event(e0)
    for _ in range(steps):
        step()
    e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return dict(ms_per_step=ms, us_per_call=ms * 1000.0 / len(calls), h2d=h2d, d2h=d2h)


def visible_key_rows(seq_lens, q_lens, H) -> int:
    """Sum over the query rows of the keys each one sees (the causal rule): the oracle's
    work is proportional to it."""
    n = 0
    for ctx, q in zip(seq_lens, q_lens):
        n += sum(int(ctx) - int(q) + i + 1 for i in range(int(q))) * H
    return n


def oracle_sample(prob, tokens: int = 1, max_keys: int | None = None):
    """A bounded sample of one call for the float64 oracle: the first `tokens` verify
    tokens of the first request, against the first `max_keys` keys of its context (all of
    them when None; token i keeps its causal key range within the sample), and the factor
    that scales the sample's time to the whole call (visible key-rows of the call over
    those of the sample)."""
    ctx, q = int(prob.seq_lens[0]), int(prob.q_lens[0])
    t = max(1, min(q, tokens))
    keys = ctx - q + t if max_keys is None else max(t, min(ctx - q + t, int(max_keys)))
    sub = inputs.Problem(H=prob.H, seq_lens=np.array([keys], np.int32), q_lens=np.array([t], np.int32),
                         page_table=prob.page_table[:1], q=prob.q[:t].clone(), kv=prob.kv, kv_dtype=prob.kv_dtype,
                         kv_scale=prob.kv_scale, sm_scale=prob.sm_scale)
    scale = visible_key_rows(prob.seq_lens, prob.q_lens, prob.H) / visible_key_rows(sub.seq_lens, sub.q_lens, prob.H)
    return sub, scale


REF_BUDGET_S = 150.0  # oracle seconds of a whole `--impl reference` run
CAL_KEYS = 16384  # keys of the calibration sample that sizes each call's timed sample
_ORACLE_RATE: dict = {}  # call name -> oracle seconds per key of one verify token


def cpu_baseline(probs, budget_s: float = 15.0):
    """The float64 oracle, as it stands (split + merge mode, 64 key chunks per request),
    on this host's cores, over a bounded sample of every call of the step: the first
    verify token of each call against the first keys of its context, as many keys as fit
    an equal share of `budget_s` seconds (a calibration sample of CAL_KEYS keys sets the
    rate), timed and scaled to the whole call by its visible key-rows."""
    import oracle

    oracle.build()
    cores = os.cpu_count() or 1

    def timed(sub):
        kvd = oracle.KV_BF16 if sub.kv_dtype == inputs.KV_BF16 else oracle.KV_FP8_E4M3
        bounds = [sorted(set(int(c) * i // 64 for i in range(65))) for c in sub.seq_lens]
        t0 = time.perf_counter()
        oracle.decode(sub.q_bits(), sub.kv_bits(), kvd, sub.kv_scale, sub.page_table, sub.page_size,
                      sub.seq_lens, sub.q_lens, sub.H, sub.sm_scale, mode=oracle.MODE_SPLIT, split_bounds=bounds,
                      nthreads=cores)
        return time.perf_counter() - t0

    us, keys = [], []
    share = budget_s / max(1, len(probs))
    for prob in probs:
        rate = _ORACLE_RATE.get(prob.name)
        if rate is None:  # once per call and process: seconds per key of one token
            cal, _ = oracle_sample(prob, 1, CAL_KEYS)
            rate = _ORACLE_RATE[prob.name] = timed(cal) / int(cal.seq_lens[0])
        sub, scale = oracle_sample(prob, 1, max(CAL_KEYS, int(share / max(rate, 1e-12))))
        keys.append(int(sub.seq_lens[0]))
        us.append(timed(sub) * 1e6 * scale)
    return dict(us_per_call=float(np.mean(us)), cores=cores, calls=len(probs),
                sample=(f"every call of the step ({len(probs)}), each on its first verify token of the first "
                        f"request against its first {min(keys)}..{max(keys)} keys (sized to ~{budget_s:.0f} s of "
                        "oracle time per step), oracle split+merge mode; time scaled to the whole call by visible "
                        "key-rows"))


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the default process group (x itself when
    there is no group or one rank)."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph-calls", type=int, default=4, choices=range(1, 65), metavar="1..64",
                    help="copies of each call, each on a cache of its own, captured back to back in the call's "
                         "CUDA graph (time per call = graph time / this)")
    ap.add_argument("--l2", default="none", choices=["flush", "none"],
                    help="none (default): rely on the step's inputs being larger than L2 (every call of a "
                         "step reads its own cache of >= 151 MB, all of them together >= 604 MB); flush: "
                         "also write 256 MB before every timed call")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")

    probs, desc = workload(args.workload)
    calls_per_step = len(probs)

    if args.impl == "reference":
        # the oracle is the reference arm: rank 0 only, bounded samples per step
        if rank != 0:
            return
        # each step a bounded sample, sized so that the whole run takes ~REF_BUDGET_S
        budget = min(30.0, max(1.0, REF_BUDGET_S / (args.warmup + args.steps)))
        times = []
        for i in range(args.warmup + args.steps):
            r = cpu_baseline(probs, budget)
            if i >= args.warmup:
                times.append(r["us_per_call"])
        v = statistics.median(times)
        line = {"metric": METRIC, "value": v, "unit": "us/call", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": v * calls_per_step / 1000.0, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {**desc, "l2": "n/a (CPU)"}, "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "us/call", "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": v, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    res = run_ours(args, probs, desc, rank, world)
    step_ms = max_over_ranks(float(np.median(res["step_ms"])), "cuda")
    # whole-job figure: every rank ran calls_per_step x graph_calls calls in step_ms
    us_per_call = step_ms * 1000.0 / (calls_per_step * args.graph_calls * world)
    hbm_peak, tf_peak, peak_src = load_peaks()
    per_call_ms = np.median(res["per_call_ms"], axis=0)
    def tensor_peak(prob):
        # the contraction's own dtype: an e4m3 cache runs e4m3 MMAs, whose dense peak is the
        # measured bf16 peak times the nominal 2x ratio
        return tf_peak * (2.0 if prob.kv_dtype == inputs.KV_FP8 else 1.0)

    traffic = profiled_traffic(os.path.join(ROOT, "profiles", f"dram_traffic_{args.workload}.md"))
    rows = []
    for c, ms in zip(res["calls"], per_call_ms):
        prob = c["prob"]
        nbytes = algorithmic_bytes(prob)
        flops = algorithmic_flops(prob)
        gbs = nbytes / (ms * 1e-3) / 1e9
        hf, tf = gbs / hbm_peak, flops / (ms * 1e-3) / 1e12 / tensor_peak(prob)
        rows.append(dict(name=prob.name, dtype=mma_dtype(prob), us=round(ms * 1000.0, 2), kv_gbs=round(gbs, 1),
                         hbm_frac=round(hf, 3), hbm_frac_rated=round(gbs / HBM_RATED_GBS, 3),
                         tensor_frac=round(tf, 3), combined_frac=round(max(hf, tf), 3),
                         traffic=traffic.get(prob.name), units=c["dec"].info["n_units"],
                         cta_pair=c["dec"].cta_pair, merge_items=c["dec"].info["n_merge"]))
    # roofline of the dominant kernel (the fold kernel, launched once per call; each timed
    # call is the whole mla_decode_run, fold + merge): the step's algorithmic bytes (or
    # flops, when the step's tensor time at peak exceeds its HBM time) over the step's call
    # time, i.e. per average launch, against the measured peak
    n_calls = len(res["calls"])
    dbytes = sum(algorithmic_bytes(c["prob"]) for c in res["calls"]) // n_calls
    dflops = sum(algorithmic_flops(c["prob"]) for c in res["calls"]) / n_calls
    t_hbm = sum(algorithmic_bytes(c["prob"]) / (hbm_peak * 1e9) for c in res["calls"])
    t_tensor = sum(algorithmic_flops(c["prob"]) / (tensor_peak(c["prob"]) * 1e12) for c in res["calls"])
    tensor_bound = t_tensor > t_hbm
    call_s = float(per_call_ms.mean()) * 1e-3
    achieved = dflops / call_s / 1e12 if tensor_bound else dbytes / call_s / 1e9
    # for a step that mixes bf16 and e4m3 calls, the peak that gives each call its own
    # dtype's peak time (sum of flops over sum of flops / peak)
    peak = round(n_calls * dflops / (t_tensor * 1e12), 1) if tensor_bound else hbm_peak
    call_traffic = [traffic.get(c["prob"].name) for c in res["calls"]]
    mean_traffic = int(sum(call_traffic) / n_calls) if all(t is not None for t in call_traffic) else None
    dtypes = sorted({mma_dtype(c["prob"]) for c in res["calls"]})
    line = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": " + ".join(dtypes), "data": "synthetic",
        "config": {**desc, "parallelism": "replicas" if world > 1 else "single",
                   "value_note": "whole job: the slowest rank's step time over the calls all ranks ran",
                   "dtype_note": "per call: the tensor-core operand type (fp32 accumulation and softmax)",
                   "l2": ("flushed before every graph replay (256 MB write)" if args.l2 == "flush" else
                          "inputs larger than L2: every call reads its own cache, "
                          f"{args.graph_calls * sum(c['prob'].kv.numel() * c['prob'].kv.element_size() for c in res['calls']) / 1e6:.0f} MB in total > 126 MB L2"),
                   "timing": (f"each call captured {args.graph_calls} times back to back in one CUDA graph (a cache "
                              "of its own per copy); CUDA events around the replay; time per call = graph time / "
                              f"{args.graph_calls}; a step replays every call's graph; median over steps"),
                   "calls_per_step": calls_per_step * args.graph_calls, "per_call": rows},
        "roofline": {"bound": "tensor" if tensor_bound else "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s" if tensor_bound else "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": mean_traffic,
                     "traffic_note": ("ncu DRAM read+write bytes of one fold launch, mean over the step's calls, "
                                      "from the committed profile when the hash of the kernel sources matches, "
                                      "else null"),
                     "algorithmic_bytes": dbytes, "algorithmic_flops": dflops,
                     "kernel": ("fold kernel (fold_decode_kernel on single CTAs, or fold_pair_kernel on clusters "
                                "of two CTAs for 49..96-row bf16 fold groups) + lse_merge_kernel, per "
                                f"mla_decode_run call, mean over the step's {n_calls} calls"),
                     "peak_source": (f"{peak_src} bf16_tflops for bf16 calls, x 2 (nominal ratio) for e4m3 calls"
                                     if tensor_bound else f"{peak_src} hbm_gbs"),
                     **({} if tensor_bound else {"peak_rated": HBM_RATED_GBS,
                                                 "frac_rated": round(achieved / HBM_RATED_GBS, 4),
                                                 "peak_rated_source": "GB300 HBM3e nominal 7.9 TB/s"})},
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "e2e": {"value": round(max_over_ranks(res["e2e"]["us_per_call"], "cuda") / world, 2), "unit": "us/call",
                "h2d_bytes_per_step": res["e2e"]["h2d"], "d2h_bytes_per_step": res["e2e"]["d2h"]},
        "device_status": res["status"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(probs)
        line["cpu_baseline"] = {"value": round(cb["us_per_call"], 1), "unit": "us/call", "cores": cb["cores"],
                                "kind": "oracle", "sample": cb["sample"]}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
