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
time over eager launches, against the measured HBM copy bandwidth).  ``e2e`` re-times the step through the public API from host
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
        "config": workload_config(w),
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
    from paged_kv_cache_313_gb300.runner import DeviceStep

    pa.lib()  # fail loudly if the CUDA library is missing
    w = W.make(args.workload, sharding.shard_seed(args.seed, rank))
    step = DeviceStep(w, dev, cascade=args.cascade)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    other = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=dev) if args.l2_flush == "write-read" else None

    def flush_l2(v):
        """Evict the step's data from L2 (outside the timed events): a 512 MiB write, then (write-read)
        a 512 MiB read of another buffer, so that the flush's dirty lines are written back here and
        not inside the next timed step."""
        flush.fill_(v)
        if other is not None:
            other.view(torch.int64).sum()  # a plain read of the 512 MiB (no widening copy)
    decode_launches = 0
    if step.use_cascade:  # decode (prefix items + tails) and merge; a separate prefix pass for groups over 32 rows
        decode_launches = 2 if w.max_group_size * (w.num_q_heads // w.num_kv_heads) <= 32 else 3
    elif w.num_decode:  # the decode kernel, plus the split-KV merge kernel when contexts span partitions
        _, splits = pa.pa_decode_plan(w.num_decode, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                      step.max_context_len)
        decode_launches = 1 + (1 if splits > 1 else 0)
    write_launches = 0 if step.fused_decode_write and not w.num_chunks else 1  # slot mapping + KV write
    launches_per_step = write_launches + decode_launches + (1 if w.num_chunks else 0)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        flush_l2(1)
        step.run()
    barrier()
    if args.graph:
        step.capture()
        for _ in range(3):
            flush_l2(1)
            step.replay()
        barrier()

    # ---- timed region: exactly K whole steps, L2 flushed before each (outside the events)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = visible.split(",")[local].strip() if visible else str(local)
    sampler = ClockSampler(smi_index)
    time.sleep(0.3)
    barrier()
    t0 = time.time()
    for i in range(K):
        flush_l2(i & 0xFF)
        ev[i][0].record(stream)
        if args.graph:
            step.replay()
        else:
            step.run()
        ev[i][1].record(stream)
    barrier()
    t1 = time.time()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # ---- per-kernel times (eager launches, same flush) for the roofline
    K1 = max(3, min(K, 100))
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K1)]
    for i in range(K1):
        e = kev[i]
        flush_l2(i & 0xFF)
        e[0].record(stream)
        step.write_stage()
        e[1].record(stream)
        step.decode_stage()
        e[2].record(stream)
        step.prefill()
        e[3].record(stream)
    barrier()
    write_ms = [e[0].elapsed_time(e[1]) for e in kev]
    decode_ms = [e[1].elapsed_time(e[2]) for e in kev]
    prefill_ms = [e[2].elapsed_time(e[3]) for e in kev]

    # ---- the same K steps back to back with no L2 flush between them (context for the flushed number:
    # whatever of the step's data is still in the 129 MB L2 is read from there)
    wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush_l2(0)
    wa.record(stream)
    for i in range(K):
        if args.graph:
            step.replay()
        else:
            step.run()
    wb.record(stream)
    barrier()
    warm_ms = wa.elapsed_time(wb) / K

    # ---- end to end through the public API: the packed inputs copied in from
    # pinned host memory (one copy), then the step, whose kernels store the
    # outputs straight into a pinned host buffer (d2h: those output bytes)
    host_in = step.pinned_inputs()
    host_out = step.pinned_outputs()
    step.step_from_host(host_in, host_out)
    if args.graph:
        step.capture_from_host(host_in, host_out)
    barrier()
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    K2 = max(1, min(K, 50))
    for i in range(K2):
        flush_l2(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step.run_from_host(host_in, host_out, graph=args.graph)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    sampler.stop()
    errors = step.errors()

    mean_step, mean_dec, mean_e2e, median_step, warm_step = sharding.max_over_ranks(
        [statistics.mean(step_ms), statistics.mean(decode_ms), statistics.mean(e2e_ms), statistics.median(step_ms),
         warm_ms], device=dev)

    hbm, bf16_tf, bf16_tf_sus, peak_kind = peaks()
    alg_bytes = decode_algorithmic_bytes(w)  # each physical K/V slot once
    if step.fused_decode_write:  # the decode tokens' new K/V rows: read from k_new/v_new, written to the pools
        alg_bytes += 2 * w.num_decode * w.kv_bytes_per_token()
    logical_bytes = decode_algorithmic_bytes(w, unique=False)  # every sequence's whole context
    achieved = alg_bytes / (mean_dec * 1e-3) / 1e9
    tokens = sharding.total_units(w.num_decode)
    value = tokens / (mean_step * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": mean_step, "ms_per_step_median": median_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 KV, bf16 q" if w.kv_fp8 else "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": workload_config(w, args.l2_flush),
        "kv_read_gbs": (sum(int(x) for x in w.context_lens[: w.num_decode]) * w.kv_bytes_per_token() * world)
                       / (mean_step * 1e-3) / 1e9,
        "roofline": {"bound": "hbm",
                     "kernel": ("pa_decode_cascade (decode_tc_kernel: shared-prefix items + tails; "
                                "decode_merge_kernel)" if step.use_cascade
                                else "pa_decode_fp8 (decode_tc_kernel over e4m3 pools + decode_merge_kernel)"
                                if w.kv_fp8
                                else "pa_decode_write (decode_tc_kernel with the decode tokens' KV write + "
                                     "decode_merge_kernel)" if step.fused_decode_write
                                else "pa_decode (decode_tc_kernel + decode_merge_kernel)"),
                     "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "algorithmic_bytes_per_launch": alg_bytes, "ms_per_launch": mean_dec,
                     "logical_bytes_per_launch": logical_bytes,
                     "effective_gbs": logical_bytes / (mean_dec * 1e-3) / 1e9,
                     "traffic": recorded_traffic("pa_decode", w.name)},
        "stage_ms": {"kv_write (separate launch)": statistics.mean(write_ms), "decode": mean_dec,
                     "prefill": statistics.mean(prefill_ms)},
        "e2e": {"value": tokens / (mean_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": mean_e2e, "steps": K2,
                "launch": "cuda_graph" if args.graph else "eager"},
        "warm_l2": {"value": tokens / (warm_step * 1e-3), "unit": "tokens/s", "ms_per_step": warm_step, "steps": K,
                    "note": "the same step repeated with no L2 flush between steps"},
        "step_launch": "cuda_graph" if args.graph else "eager",
        "gpu_launches": K * launches_per_step,
        "kv_memory": kv_memory(w),
        "clocks": sampler.summary(t0, t1),
        "device_errors": errors,
    }
    if w.num_chunks:
        fl = prefill_flops(w)
        pm = statistics.mean(prefill_ms)
        line["prefill"] = {"flops_per_launch": fl, "ms_per_launch": pm, "achieved_tflops": fl / (pm * 1e-3) / 1e12,
                           "peak_tflops": bf16_tf, "frac": fl / (pm * 1e-3) / 1e12 / bf16_tf}
    if rank == 0 and not args.no_cpu_baseline:
        per, n, threads = oracle_step_time(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": w.num_decode / per, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "nproc": os.cpu_count(),
                                "sample": f"{n} full oracle steps of workload {w.name} (fp64 C, {threads} threads)"}
        if w.name in SINGLE_THREAD_ORACLE and threads > 1:
            per1, n1, _ = oracle_step_time(w, min(5.0, args.cpu_seconds), threads=1)
            line["cpu_baseline"]["single_thread"] = {
                "value": w.num_decode / per1, "unit": "tokens/s", "cores": 1,
                "sample": f"{n1} full oracle steps of workload {w.name} (fp64 C, 1 thread)"}
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
