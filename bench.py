"""Benchmark of the paged-attention hot path on GB300.

One step = one pass of the whole hot path over one batch: slot mapping and KV
write for every new token of the step, then paged decode (and, for the mixed
workload, causal chunked prefill).  Default workload: 64 decode sequences,
32 query / 8 KV heads, head_dim 128, block_size 16, context lengths U[128,4096],
bf16, random non-contiguous block tables.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line (rank 0).  ``value`` is decode tokens/s (one token per
sequence per step) over all ranks, timed over exactly K steps, each a replay
of the step captured as a CUDA graph (``--no-graph``: eager launches).  The
roofline object describes the pa_decode call — the decode kernel and its
split-KV merge kernel — (algorithmic K/V bytes per call / its CUDA-event
time over eager launches after the L2 flush, against the measured HBM copy
bandwidth).  The line also carries a
sustained leg (the headline step, flushed, back to back for about 1.5 s, with
the clock samples taken during it) and, under ``workloads``, the same
measurements for every other configuration at ``--sweep-steps`` steps each,
with an oracle sample per configuration.  ``e2e`` re-times the step through the public API from host
memory: the step's packed inputs copied in from pinned memory (one copy), the
step (graph replay unless ``--no-graph``), the packed outputs copied back (one
copy), all inside the events.
L2 is flushed before every timed step: a 512 MiB write, then (default
``--l2-flush write-read``) a 512 MiB read of another buffer, so that the
write's dirty lines are written back before the timed step rather than
inside it.  Under torchrun each
rank runs an independent shard with its own seed (weak scaling, no collective
on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode KV-read GB/s (% of HBM peak) and decode tokens/s on 1 GB300"
DEFAULT_WORKLOAD = "decode_bf16"
FLUSH_BYTES = 512 << 20
# workloads whose oracle is also timed on one thread (the small correctness case and the default decode batch)
SINGLE_THREAD_ORACLE = ("tiny_fp32", "decode_bf16")
# the configurations measured after the headline (each at --sweep-steps), reported under "workloads"
SWEEP = ("tiny_fp32", "decode_bf16", "longctx_bf16", "shared_prefix_bf16", "mixed_bf16", "decode_fp8")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", choices=["write", "write-read"], default="write-read",
                    help="between timed steps: write 512 MiB, and (write-read) then read another 512 MiB so "
                         "that no dirty flush lines are written back inside a timed step")
    ap.add_argument("--no-cascade", dest="cascade", action="store_false",
                    help="plain paged decode even where decode sequences share prefixes")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch the timed steps eagerly instead of replaying a captured CUDA graph")
    ap.add_argument("--sustained-seconds", type=float, default=1.5,
                    help="after the K timed steps, flushed steps back to back for this long (clock samples)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="measure only the headline workload (default: also every other configuration)")
    ap.add_argument("--sweep-steps", type=int, default=20, help="timed steps per configuration of the sweep")
    ap.add_argument("--sweep-cpu-seconds", type=float, default=4.0,
                    help="target CPU time of each sweep configuration's oracle sample (at least one full step)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha256_16") == source_digest(d["source_files"]):
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms with host timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        window = [p for t, p in self.samples if t0 <= t <= t1]
        scope = "timed"
        if len(window) < 3:
            window = [p for t, p in self.samples if t <= t1 + 1.0]
            scope = "run"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in window if num(p[0]) is not None]
        mx = [num(p[1]) for p in window if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in window for n, v in zip(names, p[4:8]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(window), "window": scope}


def decode_kv_tokens(w):
    """(unique, logical) K/V token slots the decode step reads: logical counts
    every sequence's whole context; unique counts each physical slot once (a
    block shared by several sequences is read once by an ideal kernel)."""
    import numpy as np

    nd, B = w.num_decode, w.block_size
    ctx = np.asarray(w.context_lens[:nd], dtype=np.int64)
    tables = np.asarray(w.block_tables[:nd], dtype=np.int64)
    filled = {}  # physical block -> valid slots [0, n) read by some sequence
    for s in range(nd):
        L = int(ctx[s])
        nb = -(-L // B)
        for b in range(nb):
            pb = int(tables[s, b])
            n = min(B, L - b * B)
            if filled.get(pb, 0) < n:
                filled[pb] = n
    return sum(filled.values()), int(ctx.sum())


def decode_algorithmic_bytes(w, unique: bool = True) -> int:
    """Bytes the decode kernel must move: K and V of every valid context token
    (each physical slot once when `unique`), the queries and outputs, the
    block-table entries in use and the lengths."""
    nd = w.num_decode
    ctx = [int(x) for x in w.context_lens[:nd]]
    uniq, logical = decode_kv_tokens(w)
    kv = (uniq if unique else logical) * w.kv_bytes_per_token()
    qo = 2 * nd * w.num_q_heads * w.head_dim * w.elem_bytes
    tables = sum(-(-L // w.block_size) for L in ctx) * 4 + nd * 4
    return kv + qo + tables


def prefill_flops(w) -> float:
    """Causal attention flops of the chunks: 4*D*Hq per (query, visible key)."""
    tot = 0
    for c in range(w.num_chunks):
        n = int(w.cu_q_lens[c + 1] - w.cu_q_lens[c])
        off = int(w.q_start_pos[c])
        tot += n * off + n * (n + 1) // 2
    return 4.0 * w.head_dim * w.num_q_heads * tot


def kv_memory(w):
    """Per-request KV footprint and fragmentation of the workload's block tables
    next to a contiguous max-length reservation (host-side measurement)."""
    from paged_kv_cache_313_gb300.memstats import utilisation

    if w.allocator is None:
        return None
    u = utilisation(w.allocator, w.seq_ids, w.kv_bytes_per_token())
    keep = ("per_request_bytes_mean", "per_request_bytes_p95", "pool_bytes_used", "fragmentation",
            "max_tail_waste_slots", "contiguous_reserved_bytes", "contiguous_waste")
    return {k: u[k] for k in keep}


# ---------------------------------------------------------- CPU oracle arm
def oracle_step_time(w, target_seconds: float, threads: int | None = None):
    """Time the oracle's full step (slot mapping, KV write, decode, prefill) on
    the host cores (all of them unless `threads` is given), repeating until
    target_seconds of CPU time have passed."""
    import numpy as np

    import oracle
    from paged_kv_cache_313_gb300.workloads import storage_numpy

    threads = threads or os.cpu_count() or 1
    bt = w.block_tables.numpy()
    kc0 = storage_numpy(w.k_cache)
    vc0 = storage_numpy(w.v_cache)
    args = dict(kn=storage_numpy(w.k_new), vn=storage_numpy(w.v_new), qd=storage_numpy(w.q_decode),
                qp=storage_numpy(w.q_prefill))
    kc, vc = kc0.copy(), vc0.copy()
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        slots, _ = oracle.slot_mapping(bt, w.seq_idx.numpy(), w.pos.numpy(), w.block_size, w.num_blocks)
        nd = w.num_decode
        if w.kv_fp8:  # quantising write, then attention over the pools read back in float64
            oracle.write_kv_fp8(args["kn"], args["vn"], kc, vc, slots, w.k_scale, w.v_scale)
            if nd:
                oracle.decode(w.q_decode.double().numpy(), oracle.dequant_e4m3(kc, w.k_scale),
                              oracle.dequant_e4m3(vc, w.v_scale), bt[:nd], w.context_lens.numpy()[:nd], w.scale,
                              num_threads=threads)
        else:
            oracle.write_kv(args["kn"], args["vn"], kc, vc, slots)
        if nd and not w.kv_fp8:
            oracle.decode(args["qd"], kc, vc, bt[:nd], w.context_lens.numpy()[:nd], w.scale, num_threads=threads)
        if w.num_chunks:
            oracle.prefill(args["qp"], w.cu_q_lens.numpy(), w.q_start_pos.numpy(), w.seq_of_chunk.numpy(), kc, vc, bt,
                           w.context_lens.numpy(), w.scale, num_threads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= target_seconds or len(times) >= 1000:
            break
    del np
    return statistics.mean(times), len(times), threads


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_313_gb300 import workloads as W

    w = W.make(args.workload, args.seed)
    steps = max(1, args.steps)
    # every step is one oracle pass over the full workload; bounded so the run ends within minutes
    budget = min(max(args.cpu_seconds, 1.0), 120.0)
    per_step, n, threads = oracle_step_time(w, budget / max(1, min(steps, 4)))
    tokens = w.num_decode
    value = tokens / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.l2_flush),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} full oracle steps of workload {w.name} (fp64 C, {threads} threads)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, l2_flush: str = "write"):
    ctx = [int(x) for x in w.context_lens[: w.num_decode]]
    cfg = {"workload": w.name, "decode_seqs": w.num_decode, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
           "head_dim": w.head_dim, "block_size": w.block_size, "num_blocks": w.num_blocks,
           "sum_context_tokens": sum(ctx), "max_context": max(ctx) if ctx else 0,
           "prefill_chunks": w.num_chunks, "prefill_queries": int(w.cu_q_lens[-1]) if w.num_chunks else 0,
           "new_tokens": int(w.seq_idx.numel()), "seed": w.meta.get("seed", 0),
           "l2": "flushed before every timed step (512 MiB write)"}
    if l2_flush == "write-read":
        cfg["l2"] = ("flushed before every timed step: 512 MiB write, then a 512 MiB read of another buffer "
                     "(dirty flush lines written back outside the timed events)")
    shared = int((w.prefix_lens > 0).sum()) if w.num_decode else 0
    if shared:
        cfg["shared_prefix_seqs"] = shared
        cfg["groups"] = int(len(w.group_offsets) - 1)
    if w.kv_fp8:
        cfg["kv_pool"] = f"e4m3, k_scale {w.k_scale:g}, v_scale {w.v_scale:g}"
    return cfg


# ------------------------------------------------------------- native arm
def launches_per_step(step, w, pa):
    """Our kernels per step: the fused slot mapping + KV write (unless the decode kernel writes every new token
    itself), the decode kernel(s) and the split-KV merge, and the prefill kernel."""
    decode_launches = 0
    if step.use_cascade:  # decode (prefix items + tails) and merge; a separate prefix pass for groups over 32 rows
        decode_launches = 2 if w.max_group_size * (w.num_q_heads // w.num_kv_heads) <= 32 else 3
    elif w.num_decode:  # the decode kernel, plus the split-KV merge kernel when contexts span partitions
        _, splits = pa.pa_decode_plan(w.num_decode, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                      step.max_context_len)
        decode_launches = 1 + (1 if splits > 1 else 0)
    write_launches = 0 if step.fused_decode_write and not w.num_chunks else 1
    return write_launches + decode_launches + (1 if w.num_chunks else 0)


def decode_kernel_name(step, w):
    if step.use_cascade:
        return "pa_decode_cascade (decode_tc_kernel: shared-prefix items + tails; decode_merge_kernel)"
    if w.kv_fp8 and step.fused_decode_write:
        return ("pa_decode_write_fp8 (decode_tc_kernel over e4m3 pools with the decode tokens' quantising write + "
                "decode_merge_kernel)")
    if w.kv_fp8:
        return "pa_decode_fp8 (decode_tc_kernel over e4m3 pools + decode_merge_kernel)"
    if step.fused_decode_write:
        return "pa_decode_write (decode_tc_kernel with the decode tokens' KV write + decode_merge_kernel)"
    if w.dtype.is_floating_point and w.elem_bytes == 4:
        return "pa_decode (decode_fma_kernel, fp32 + decode_merge_kernel)"
    return "pa_decode (decode_tc_kernel + decode_merge_kernel)"


class Flusher:
    """Evicts the step's data from L2 between timed steps (outside the events): a 512 MiB write, then
    (write-read) a 512 MiB read of another buffer, so that the flush's dirty lines are written back before
    the next timed step and not inside it."""

    def __init__(self, torch, dev, mode):
        self.buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        other = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=dev) if mode == "write-read" else None
        self.other = other.view(torch.int64) if other is not None else None

    def __call__(self, v):
        self.buf.fill_(v)
        if self.other is not None:
            self.other.sum()  # a plain read of the 512 MiB (no widening copy)


def measure(w, args, dev, flush, K, graph=True, sustained_s=0.0, sampler=None, barrier=None):
    """Time one workload's step on the device: K flushed steps (graph replays), the decode call and the prefill
    call alone (eager, flushed) for the roofline, K steps with a warm L2, the step end to end from pinned host
    memory, and optionally a sustained leg of back-to-back flushed steps lasting `sustained_s` seconds.
    Returns a dict of results (per rank; the caller takes the max over ranks)."""
    import torch

    from paged_kv_cache_313_gb300 import pa
    from paged_kv_cache_313_gb300.runner import DeviceStep

    step = DeviceStep(w, dev, cascade=args.cascade)
    stream = torch.cuda.current_stream(dev)
    sync = barrier or (lambda: torch.cuda.synchronize(dev))
    for _ in range(max(3, args.warmup)):
        flush(1)
        step.run()
    sync()
    if graph:
        step.capture()
        for _ in range(3):
            flush(1)
            step.replay()
        sync()

    def timed_steps(n, flush_each=True):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            if flush_each:
                flush(i & 0xFF)
            ev[i][0].record(stream)
            if graph:
                step.replay()
            else:
                step.run()
            ev[i][1].record(stream)
        return ev

    # ---- timed region: exactly K whole steps, L2 flushed before each (outside the events)
    sync()
    t0 = time.time()
    ev = timed_steps(K)
    sync()
    t1 = time.time()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # ---- per-stage times for the roofline: eager launches between events, same flush.  After the flush the
    # GPU spins for a while (a device-side sleep) so that the host has enqueued every stage before the first
    # event is reached: no host launch gap falls inside a stage's interval (without it, a short kernel in front
    # of the decode call left the decode's interval up to 15 % long on some runs)
    K1 = max(3, min(K, 100))
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K1)]
    for i in range(K1):
        e = kev[i]
        flush(i & 0xFF)
        torch.cuda._sleep(400_000)  # ~0.2 ms of GPU cycles, outside the events
        e[0].record(stream)
        step.write_stage()
        e[1].record(stream)
        step.decode_stage()
        e[2].record(stream)
        step.prefill()
        e[3].record(stream)
    sync()
    write_ms = [e[0].elapsed_time(e[1]) for e in kev]
    decode_ms = [e[1].elapsed_time(e[2]) for e in kev]
    prefill_ms = [e[2].elapsed_time(e[3]) for e in kev]

    # ---- the same K steps back to back with no L2 flush between them (context for the flushed number)
    wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush(0)
    wa.record(stream)
    for _ in range(K):
        if graph:
            step.replay()
        else:
            step.run()
    wb.record(stream)
    sync()
    warm_ms = wa.elapsed_time(wb) / K

    # ---- sustained: flushed steps back to back for at least sustained_s seconds, so that clock samples
    # (every 100 ms) fall inside the measured work
    sustained = None
    if sustained_s > 0:
        per = statistics.mean(step_ms) + 0.2  # the flush between steps takes about 0.2 ms
        n = max(K, int(sustained_s * 1e3 / per) + 1)
        sync()
        s0 = time.time()
        sev = timed_steps(n)
        sync()
        s1 = time.time()
        sms = [a.elapsed_time(b) for a, b in sev]
        sustained = {"steps": n, "ms_per_step": statistics.mean(sms), "wall_s": s1 - s0,
                     "clocks": sampler.summary(s0, s1) if sampler else None}

    # ---- end to end through the public API: the packed inputs copied in from pinned host memory (one
    # copy), then the step, whose kernels store the outputs into a pinned host buffer (d2h: those bytes)
    host_in = step.pinned_inputs()
    host_out = step.pinned_outputs()
    step.step_from_host(host_in, host_out)
    if graph:
        step.capture_from_host(host_in, host_out)
    sync()
    e2e_ms = []
    K2 = max(1, min(K, 50))
    for i in range(K2):
        flush(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step.run_from_host(host_in, host_out, graph=graph)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    errors = step.errors()
    res = {"step": step, "step_ms": step_ms, "decode_ms": decode_ms, "write_ms": write_ms,
           "prefill_ms": prefill_ms, "warm_ms": warm_ms, "e2e_ms": e2e_ms, "K2": K2, "t0": t0, "t1": t1,
           "h2d": host_in.numel() * host_in.element_size(), "d2h": host_out.numel() * host_out.element_size(),
           "errors": errors, "sustained": sustained, "launches_per_step": launches_per_step(step, w, pa)}
    return res


def roofline_of(w, step, mean_dec, hbm, peak_kind):
    alg_bytes = decode_algorithmic_bytes(w)  # each physical K/V slot once
    if step.fused_decode_write:  # the decode tokens' new K/V rows: read from k_new/v_new, written to the pools
        # (e4m3 pools: the rows are read as bf16, twice the bytes of the codes written)
        alg_bytes += (3 if w.kv_fp8 else 2) * w.num_decode * w.kv_bytes_per_token()
    logical_bytes = decode_algorithmic_bytes(w, unique=False)  # every sequence's whole context
    achieved = alg_bytes / (mean_dec * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": decode_kernel_name(step, w), "achieved": achieved, "peak": hbm,
            "unit": "GB/s", "frac": achieved / hbm, "peak_kind": f"{peak_kind} hbm_gbs (copy)",
            "algorithmic_bytes_per_launch": alg_bytes, "ms_per_launch": mean_dec,
            "logical_bytes_per_launch": logical_bytes, "effective_gbs": logical_bytes / (mean_dec * 1e-3) / 1e9,
            "traffic": recorded_traffic("pa_decode", w.name)}


def prefill_of(w, prefill_ms, bf16_tf, peak_kind):
    fl = prefill_flops(w)
    pm = statistics.mean(prefill_ms)
    return {"kernel": "prefill_tc_kernel", "bound": "tensor", "flops_per_launch": fl, "ms_per_launch": pm,
            "achieved_tflops": fl / (pm * 1e-3) / 1e12, "peak_tflops": bf16_tf,
            "frac": fl / (pm * 1e-3) / 1e12 / bf16_tf, "peak_kind": f"{peak_kind} bf16_tflops (burst)"}


def cpu_baseline_of(w, seconds, single_thread=False):
    per, n, threads = oracle_step_time(w, seconds)
    out = {"value": w.num_decode / per, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "nproc": os.cpu_count(),
           "sample": f"{n} full oracle step(s) of workload {w.name} (fp64 C, {threads} threads)"}
    if single_thread and threads > 1:
        per1, n1, _ = oracle_step_time(w, min(5.0, seconds), threads=1)
        out["single_thread"] = {"value": w.num_decode / per1, "unit": "tokens/s", "cores": 1,
                                "sample": f"{n1} full oracle step(s) of workload {w.name} (fp64 C, 1 thread)"}
    return out


def run_native(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_cache_313_gb300 import pa, sharding
    from paged_kv_cache_313_gb300 import workloads as W

    pa.lib()  # fail loudly if the CUDA library is missing
    flush = Flusher(torch, dev, args.l2_flush)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = visible.split(",")[local].strip() if visible else str(local)
    sampler = ClockSampler(smi_index)
    time.sleep(0.3)
    hbm, bf16_tf, bf16_tf_sus, peak_kind = peaks()

    # ---- the headline workload: K steps, as the contract times them, then a sustained leg
    w = W.make(args.workload, sharding.shard_seed(args.seed, rank))
    K = args.steps
    r = measure(w, args, dev, flush, K, graph=args.graph, sustained_s=args.sustained_seconds, sampler=sampler,
                barrier=barrier)
    step = r["step"]
    sus = r["sustained"]
    mean_step, mean_dec, mean_e2e, median_step, warm_step, sus_step = sharding.max_over_ranks(
        [statistics.mean(r["step_ms"]), statistics.mean(r["decode_ms"]), statistics.mean(r["e2e_ms"]),
         statistics.median(r["step_ms"]), r["warm_ms"], sus["ms_per_step"] if sus else 0.0], device=dev)
    tokens = sharding.total_units(w.num_decode)
    value = tokens / (mean_step * 1e-3)
    clocks = (sus or {}).get("clocks") or sampler.summary(r["t0"], r["t1"])
    if clocks is not None and sus is not None:
        clocks["window"] = "sustained leg (the headline step, flushed, back to back)"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": mean_step, "ms_per_step_median": median_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 KV, bf16 q" if w.kv_fp8 else "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": workload_config(w, args.l2_flush),
        "kv_read_gbs": (sum(int(x) for x in w.context_lens[: w.num_decode]) * w.kv_bytes_per_token() * world)
                       / (mean_step * 1e-3) / 1e9,
        "roofline": roofline_of(w, step, mean_dec, hbm, peak_kind),
        "stage_ms": {"kv_write (separate launch)": statistics.mean(r["write_ms"]), "decode": mean_dec,
                     "prefill": statistics.mean(r["prefill_ms"]),
                     "how": "eager launches between events, after the flush and a device-side wait"},
        "e2e": {"value": tokens / (mean_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": mean_e2e, "steps": r["K2"],
                "launch": "cuda_graph" if args.graph else "eager"},
        "warm_l2": {"value": tokens / (warm_step * 1e-3), "unit": "tokens/s", "ms_per_step": warm_step, "steps": K,
                    "note": "the same step repeated with no L2 flush between steps"},
        "step_launch": "cuda_graph" if args.graph else "eager",
        "gpu_launches": K * r["launches_per_step"],
        "kv_memory": kv_memory(w),
        "clocks": clocks,
        "device_errors": r["errors"],
    }
    if sus is not None:
        line["sustained"] = {"value": tokens / (sus_step * 1e-3), "unit": "tokens/s", "ms_per_step": sus_step,
                             "steps": sus["steps"], "wall_s": sus["wall_s"], "clocks": sus["clocks"],
                             "note": "flushed steps back to back for about "
                                     f"{args.sustained_seconds:g} s; not part of gpu_launches"}
    if w.num_chunks:
        line["prefill"] = prefill_of(w, r["prefill_ms"], bf16_tf, peak_kind)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_of(w, args.cpu_seconds, single_thread=w.name in SINGLE_THREAD_ORACLE)
    del step, r
    torch.cuda.empty_cache()

    # ---- every other configuration of the workload list: the same measurements at fewer steps
    if args.sweep:
        per = {}
        headline_entry = {"value": value, "ms_per_step": mean_step, "roofline_frac": line["roofline"]["frac"],
                          "e2e": line["e2e"]["value"], "note": "the headline above"}
        if "cpu_baseline" in line:
            headline_entry["cpu_baseline"] = line["cpu_baseline"]["value"]
        for name in SWEEP:
            if name == w.name:
                per[name] = headline_entry
                continue
            ws = W.make(name, sharding.shard_seed(args.seed, rank))
            rs = measure(ws, args, dev, flush, args.sweep_steps, graph=args.graph)
            st = rs["step"]
            ms, md, me = sharding.max_over_ranks([statistics.mean(rs["step_ms"]), statistics.mean(rs["decode_ms"]),
                                                  statistics.mean(rs["e2e_ms"])], device=dev)
            tok = sharding.total_units(ws.num_decode)
            rf = roofline_of(ws, st, md, hbm, peak_kind)
            entry = {"value": tok / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": args.sweep_steps,
                     "config": workload_config(ws, args.l2_flush),
                     "roofline": {k: rf[k] for k in ("bound", "kernel", "achieved", "peak", "unit", "frac",
                                                     "algorithmic_bytes_per_launch", "ms_per_launch",
                                                     "logical_bytes_per_launch", "effective_gbs", "traffic")},
                     "e2e": {"value": tok / (me * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": rs["h2d"],
                             "d2h_bytes_per_step": rs["d2h"], "ms_per_step": me},
                     "gpu_launches": args.sweep_steps * rs["launches_per_step"], "device_errors": rs["errors"]}
            if ws.num_chunks:
                entry["prefill"] = prefill_of(ws, rs["prefill_ms"], bf16_tf, peak_kind)
            if rank == 0 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline_of(ws, args.sweep_cpu_seconds)
            per[name] = entry
            del st, rs, ws
            torch.cuda.empty_cache()
        line["workloads"] = per
    sampler.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
