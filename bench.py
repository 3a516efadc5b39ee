"""Benchmark: one batched paged-decode step on GB300, printed as one JSON line.

A step is the whole hot path over one batch: pa_cache_write of every
sequence's new token into the paged cache, then pa_decode (partition list,
attention over the 16-token blocks, merge of split sequences).  Default
workload: the Llama-3-70B-shaped mixed-length layer (256 sequences, 90% of
~350 tokens and 10% of ~32000, 64 query / 8 KV heads, head_dim 128, bf16).

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
                    [--variant auto|fma|mma] [--impl pa|reference]

* value      logical KV GB/s of the step (sum over sequences of
             len x kv_heads x head_dim x 2 (K,V) x 2 bytes / step time),
             inputs resident in HBM, CUDA events around exactly K steps.
* e2e        the same metric through the public API from pinned host
             buffers: host allocator (slots, table), H2D of q/k/v/slots/
             table/lens, cache write, decode, D2H of the output, per step.
* roofline   the attention kernel alone: algorithmic bytes / its average
             CUDA-event duration vs the measured HBM copy bandwidth.
* cpu_baseline  the fp64 CPU oracle on a bounded sample of the workload.
--impl reference times only that oracle (the reference arm).
Under torchrun every rank runs its own replica (weak scaling, no
collective on the data path; a barrier and a max over ranks for timing).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s and seqs·steps/s; % of GB300 HBM peak"
DESCR = {
    "llama70b": "Llama-3-70B-shaped mixed-length decode layer: 256 seqs (230 x 300+U{1..100}, "
                "26 x 30000+U{1..4000} tokens), 64 q / 8 kv heads, head_dim 128, bf16, block 16",
    "llama8b": "Llama-3-8B-shaped decode layer: 64 seqs U{128..2048} tokens, 32 q / 8 kv heads, "
               "head_dim 128, bf16, block 16",
    "long": "long-context decode: 8 seqs x 32768 tokens, 32 q / 8 kv heads, head_dim 128, bf16, "
            "512-token partitions + merge",
    "tiny": "tiny decode: 4 seqs {1,17,33,100}, 4 q / 2 kv heads, head_dim 64, fp16",
    "fullstep": "full decode step: 32 layers of the Llama-3-8B shape, 128 seqs in 4 groups of 32 "
                "sharing a 1024-token prefix (ref-counted blocks), lens 1024+U{256..7168}, bf16",
}
DESCR["chunked"] = ("chunked prefill, Llama-3-70B-shaped layer (64 q / 8 kv heads, head_dim 128, "
                    "bf16): a 30000-token prompt prefilled in 8 pieces of 3750 tokens, each "
                    "iteration with the decode tokens of 20 chats of 300+U{1..100} tokens; one step "
                    "= the 8 iterations (pa_cache_write of the pieces + pa_prefill)")
PREFILL_METRIC = "paged chunked-prefill attention TFLOP/s (causal, dense-equivalent 4*q*k*d per head)"
COW_PAIRS, COW_POOL = 4096, 32768
DESCR["cow"] = (f"copy-on-write block copies: {COW_PAIRS} (source, destination) pairs of "
                "Llama-3-70B-shaped blocks (8 kv heads x 16 tokens x 128 dims, bf16, K and V: "
                f"64 KB per pair) in a {COW_POOL}-block pool; one step = one pa_copy_blocks call")
COW_METRIC = "paged KV copy-on-write block copy GB/s (bytes read + written)"
VARIANTS = {"auto": 0, "fma": 1, "mma": 2, "tc": 3}


# --------------------------------------------------------------------------- helpers

def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(lens, hq, hkv, d, elem=2, part_tokens=512, kv_elem=None, starts=None):
    """Bytes the attention kernel must move: K/V of every token it covers
    once per KV head, block ids, q, and either the output (one partition) or
    the fp32 partial (max, sum, head_dim values) of every partition.
    ``starts``: first token each sequence's attention kernel covers (the
    shared prefix of a grouped decode, whose partials always merge)."""
    L = np.asarray(lens, np.int64)
    st = np.zeros_like(L) if starts is None else np.asarray(starts, np.int64)
    n = L - st
    kv = int(n.sum()) * hkv * d * (elem if kv_elem is None else kv_elem) * 2
    ids = int(((n + 15) // 16).sum()) * 4
    q = len(L) * hq * d * elem
    nparts = (n + part_tokens - 1) // part_tokens
    direct = (nparts == 1) & (st == 0)
    out = int(direct.sum()) * hq * d * elem
    partial = int(nparts[~direct].sum()) * hq * (d + 2) * 4
    return kv + ids + q + out + partial


def logical_kv_bytes(lens, hkv, d, elem=2):
    """Sum over sequences of len x kv_heads x head_dim x 2 (K, V) x bytes."""
    return int(np.asarray(lens, np.int64).sum()) * hkv * d * elem * 2


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons), stamped on arrival."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.err = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.err = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": self.err}
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not win:
            win = [p for (_, p) in self.samples]
            note = "timed region shorter than the sampling period: samples around it"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        pw = [num(p[3]) for p in win if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(win), "note": note}


def reduce_max(value, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds_max):
    """Whole-job rate: every rank processes the same number of units (weak
    scaling), the job takes as long as its slowest rank."""
    return units_per_rank * world / seconds_max


def cpu_model():
    """Host CPU model (lscpu's "Model name", else /proc/cpuinfo), for the
    record of where the oracle baseline ran."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def gpu_identity(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        items = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(items):
            return items[local_rank]
    return str(local_rank)


# --------------------------------------------------------------------------- CPU oracle

REF_RUN_S = 150.0   # default oracle time of a whole reference-arm run (warm-up + timed steps), s


def ref_step_budget(args):
    """Seconds of oracle work per reference-arm step, so that the whole
    ``--steps K --warmup W`` run stays within ``--ref-seconds`` whatever K and
    W are."""
    return args.ref_seconds / max(1, args.steps + args.warmup)


def oracle_sample_rows(lens, n_long):
    """Rows of the workload keeping its short/long mix: n_long of the long
    sequences and 9 x n_long of the short ones (all when the mix is flat)."""
    lens = np.asarray(lens)
    med = np.median(lens)
    long_rows = np.flatnonzero(lens > 10 * med)
    short_rows = np.flatnonzero(lens <= 10 * med)
    if len(long_rows) == 0:
        return short_rows[:max(1, n_long)]
    return np.concatenate([long_rows[:n_long], short_rows[:9 * n_long]])


def time_oracle(workload, rows, threads, seed=0):
    import oracle
    from paged_kv_cache_blocks_gb300 import workloads as W
    lens = W.workload_lengths(workload, seed)[rows]
    b = W.make_batch(workload, seed=seed, poison=False, lens_override=lens.tolist())
    w = b.workload
    kc, vc = W.place_new_tokens(b, 0)
    q = b.layers[0].q.numpy().view(np.uint16)
    kc, vc = kc.numpy().view(np.uint16), vc.numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.decode(q, kc, vc, b.block_tables, b.seq_lens, w.scale, w.dtype, threads=threads)
    dt = time.perf_counter() - t0
    return dt, lens, b


def cpu_baseline(workload, budget_s=12.0):
    import oracle
    oracle.build()
    from paged_kv_cache_blocks_gb300 import workloads as W
    threads = len(os.sched_getaffinity(0))
    w = W.WORKLOADS[workload]
    lens_all = W.workload_lengths(workload, 0)
    rows = oracle_sample_rows(lens_all, 1)
    t1, lens, _ = time_oracle(workload, rows, threads)
    n_long = 1
    has_long = (np.asarray(lens_all) > 10 * np.median(lens_all)).any()
    if has_long:
        n_long = int(max(1, min(int((np.asarray(lens_all) > 10 * np.median(lens_all)).sum()),
                                round(budget_s / max(t1, 1e-3)))))
        rows = oracle_sample_rows(lens_all, n_long)
        t1, lens, _ = time_oracle(workload, rows, threads)
    kvb = logical_kv_bytes(lens, w.num_kv_heads, w.head_dim)
    # one thread, on the first long and the first short sequence of the sample
    rows1 = oracle_sample_rows(lens_all, 1)[:2]
    t_one, lens_one, _ = time_oracle(workload, rows1, 1)
    one = logical_kv_bytes(lens_one, w.num_kv_heads, w.head_dim) / t_one / 1e9
    return {"value": kvb / t1 / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": t1, "seqs_steps_per_s": len(lens) / t1,
            "single_thread_value": one,
            "single_thread_sample": f"{len(lens_one)} sequences ({int(np.sum(lens_one))} tokens), 1 thread",
            "sample": f"{len(lens)} of the {len(lens_all)} sequences of the same workload "
                      f"({int((np.asarray(lens) > 10 * np.median(lens_all)).sum())} long, same "
                      f"length draw), {int(np.sum(lens))} tokens, one decode step, fp64, "
                      f"{threads} OpenMP threads; excludes input generation"}


def prefill_flops(lens, pieces, hq, d):
    """Causal attention FLOPs of a multi-query batch: 2 (QK) + 2 (PV) per
    (query token, visible key, head, dim)."""
    total = 0
    for L, n in zip(np.asarray(lens, np.int64), np.asarray(pieces, np.int64)):
        # query j sees L - n + j + 1 keys
        total += int(n * (L - n) + n * (n + 1) // 2)
    return 4 * total * hq * d


class PrefillOracleSample:
    """One iteration of the chunked workload (by default the last, whose rows
    are the most expensive) set up once for the fp64 oracle; ``run(n_rows)``
    times it on ``n_rows`` query rows spread over the prompt piece and scales
    to FLOP/s."""

    def __init__(self, threads=None, seed=0, iteration=None):
        import oracle
        oracle.build()
        from paged_kv_cache_blocks_gb300 import workloads as W
        self.oracle = oracle
        self.threads = threads or len(os.sched_getaffinity(0))
        self.iteration = iteration or W.CHUNK_PIECES
        self.pb = W.make_prefill_batch("chunked", seed=seed, iteration=self.iteration,
                                       poison=False)
        kc, vc = self.pb.placed_pools()
        self.q = self.pb.q.numpy().view(np.uint16)
        self.kc, self.vc = kc.numpy().view(np.uint16), vc.numpy().view(np.uint16)
        self.n = int(self.pb.pieces[0])

    def run(self, n_rows):
        pb, w = self.pb, self.pb.workload
        rows = np.linspace(0, self.n - 1, n_rows).astype(np.int64)
        t0 = time.perf_counter()
        self.oracle.prefill(self.q, self.kc, self.vc, pb.block_tables, pb.seq_lens, pb.q_offsets,
                            w.scale, w.dtype, rows=rows, threads=self.threads)
        dt = time.perf_counter() - t0
        base = int(pb.seq_lens[0]) - self.n
        fl = sum(4 * (base + int(r) + 1) * w.num_q_heads * w.head_dim for r in rows)
        return fl / dt / 1e12, dt, (f"{n_rows} query tokens of piece {self.iteration} of 8 of the "
                                    f"30000-token prompt (positions {base + rows[0]}.."
                                    f"{base + rows[-1]}, all 64 heads), fp64, "
                                    f"{self.threads} OpenMP threads")


def prefill_cpu_baseline(threads=None, n_rows=None, seed=0, budget_s=12.0):
    """The fp64 oracle on query rows of the last iteration's prompt piece,
    scaled to FLOP/s; ``n_rows=None`` sizes the sample to about ``budget_s``
    seconds from an 8-row probe."""
    smp = PrefillOracleSample(threads, seed)
    if n_rows is None:
        _, sec, _ = smp.run(8)
        n_rows = int(max(8, min(3750, round(8 * budget_s / max(sec, 1e-3)))))
    v, dt, sample = smp.run(n_rows)
    return v, dt, smp.threads, sample


def run_prefill(args, rank, world, local_rank):
    """The chunked-prefill workload: one step = the 8 iterations of the
    prompt, each pa_cache_write of the iteration's new tokens + pa_prefill."""
    from paged_kv_cache_blocks_gb300 import build as pb_build
    pb_build.build()
    from paged_kv_cache_blocks_gb300 import binding as pa
    from paged_kv_cache_blocks_gb300 import workloads as W
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = W.WORKLOADS["chunked"]
    dt = torch.bfloat16
    its = []
    flops = 0
    q_tokens = 0
    for k in range(1, W.CHUNK_PIECES + 1):
        b = W.make_prefill_batch("chunked", seed=rank, iteration=k, poison=False, device="cuda")
        ws = torch.empty(pa.pa_prefill_workspace_bytes(len(b.seq_lens), b.num_q_tokens,
                                                       w.num_q_heads, w.num_kv_heads),
                         dtype=torch.uint8, device=dev)
        its.append(dict(q=b.q.view(dt), kc=b.k_cache.view(dt), vc=b.v_cache.view(dt),
                        nk=b.new_k.view(dt), nv=b.new_v.view(dt),
                        slots=torch.from_numpy(b.slot_mapping).to(dev),
                        tab=torch.from_numpy(b.block_tables).to(dev),
                        lens=torch.from_numpy(b.seq_lens).to(dev),
                        qoff=torch.from_numpy(b.q_offsets).to(dev), ws=ws,
                        out=torch.empty_like(b.q.view(dt)), msl=int(b.seq_lens.max()), host=b))
        flops += prefill_flops(b.seq_lens, b.pieces, w.num_q_heads, w.head_dim)
        q_tokens += b.num_q_tokens
    stream = torch.cuda.current_stream()

    def step(evs=None):
        for i, it in enumerate(its):
            pa.pa_cache_write(it["nk"], it["nv"], it["slots"], it["kc"], it["vc"])
            pa.pa_prefill(it["q"], it["kc"], it["vc"], it["tab"], it["lens"], it["qoff"], w.scale,
                          max_seq_len=it["msl"], out=it["out"], workspace=it["ws"],
                          events=evs[i] if evs else None, variant=VARIANTS[args.variant])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for it in its:
        bits = pa.pa_decode_check(it["ws"])
        if bits:
            raise RuntimeError(f"device error bits {bits} during warm-up")
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in its] for _ in range(args.steps)]
    for row in ev:
        for a, z in row:
            a.record(stream)
            z.record(stream)
    sampler = ClockSampler(gpu_identity(local_rank)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_host0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    stop.record(stream)
    barrier()
    t_host1 = time.time()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    ms_step = reduce_max(start.elapsed_time(stop) / args.steps, dist, dev)
    kern_ms = sum(statistics.fmean(a.elapsed_time(z) for row in ev for a, z in [row[i]])
                  for i in range(len(its)))
    tflops = job_throughput(flops, world, ms_step * 1e-3) / 1e12
    achieved = flops / (kern_ms * 1e-3) / 1e12
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
    peak_src = "measured bf16_tflops_sustained (cuBLAS bf16, seconds-long loop)" if peaks \
        else "fallback 1.7 PFLOP/s sustained"

    e2e = None
    if not args.no_e2e:
        e2e = run_prefill_e2e(args, pa, its, w, dev, barrier, dist, world, flops)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, sec, cores, sample = prefill_cpu_baseline()
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "seconds": sec,
               "sample": sample}
    line = {
        "metric": PREFILL_METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": DESCR["chunked"], "iterations": len(its),
                   "query_tokens_per_step": q_tokens, "flops_per_step": flops,
                   "kv_tokens_last_iteration": int(its[-1]["host"].seq_lens.sum()),
                   "variant": args.variant,
                   "l2": "K/V per iteration <= 155 MB, re-read by every 16-token query tile: "
                         "compute-bound; no flush",
                   "parallelism": f"replicas x{world}"},
        "query_tokens_per_s": job_throughput(q_tokens, world, ms_step * 1e-3),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": load_traffic("chunked", args.variant),
                     "traffic_per": "step (the 8 prefill launches)",
                     "kernel": "prefill_kernel (mma.sync)" if args.variant == "mma"
                     else "prefill_tc_kernel (tcgen05)",
                     "kernel_ms": kern_ms, "algorithmic_flops": flops, "peak_source": peak_src},
        "e2e": e2e,
        "gpu_launches": 3 * len(its) * args.steps,
        "clocks": sampler.summary(t_host0, t_host1) if sampler else None,
    }
    if cpu is not None:
        cpu["cpu_model"] = cpu_model()
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


def run_prefill_e2e(args, pa, its, w, dev, barrier, dist, world, flops):
    """The 8 iterations through the public API from pinned host buffers:
    H2D of each iteration's q, new k/v, slots, table, lengths and offsets,
    cache write, prefill, D2H of the output.  The copies run on their own
    streams: iteration i+1's inputs go up while iteration i computes and
    iteration i's output comes down while i+1 computes (events order each
    buffer's reuse across steps); synchronised after the last step."""
    steps = max(1, min(args.steps, max(1, args.e2e_steps // 20)))
    host = []
    for it in its:
        h = {k: it[k].cpu().pin_memory() for k in ("q", "nk", "nv", "slots", "tab", "lens", "qoff")}
        h["out"] = torch.empty_like(it["out"], device="cpu").pin_memory()
        d = {k: torch.empty_like(it[k]) for k in ("q", "nk", "nv", "slots", "tab", "lens", "qoff")}
        host.append((h, d))
    nbytes = lambda t: t.numel() * t.element_size()
    h2d = sum(nbytes(h[k]) for h, _ in host for k in ("q", "nk", "nv", "slots", "tab", "lens", "qoff"))
    d2h = sum(nbytes(h["out"]) for h, _ in host)
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    n = len(its)
    ev_up = [torch.cuda.Event() for _ in range(n)]
    ev_done = [torch.cuda.Event() for _ in range(n)]
    ev_down = [torch.cuda.Event() for _ in range(n)]
    for e in ev_done + ev_down:
        e.record(comp)

    def one():
        for i, (h, d) in enumerate(host):
            up.wait_event(ev_done[i])          # the previous step's compute read d
            with torch.cuda.stream(up):
                for k in d:
                    d[k].copy_(h[k], non_blocking=True)
            ev_up[i].record(up)
        for i, (it, (h, d)) in enumerate(zip(its, host)):
            comp.wait_event(ev_up[i])
            comp.wait_event(ev_down[i])        # the previous step's output is down
            pa.pa_cache_write(d["nk"], d["nv"], d["slots"], it["kc"], it["vc"])
            pa.pa_prefill(d["q"], it["kc"], it["vc"], d["tab"], d["lens"], d["qoff"], w.scale,
                          max_seq_len=it["msl"], out=it["out"], workspace=it["ws"],
                          variant=VARIANTS[args.variant])
            ev_done[i].record(comp)
            down.wait_event(ev_done[i])
            with torch.cuda.stream(down):
                h["out"].copy_(it["out"], non_blocking=True)
            ev_down[i].record(down)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    barrier()
    sec = reduce_max((time.perf_counter() - t0) / steps, dist, dev)
    return {"value": job_throughput(flops, world, sec) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": sec * 1e3,
            "path": "per iteration: H2D (pinned, copy stream) q, new k/v, slots, table, lens, "
                    "offsets -> pa_cache_write -> pa_prefill -> D2H out (second copy stream); "
                    "iteration i+1's inputs go up while i computes; synchronised after the last step"}


def cow_pairs(seed):
    """Distinct source and destination blocks of the copy workload (seeded)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(4000 + int(seed))
    perm = torch.randperm(COW_POOL, generator=g).to(torch.int32)
    return perm[:COW_PAIRS].clone(), perm[COW_PAIRS:2 * COW_PAIRS].clone()


class CowOracleSample:
    """``pairs`` block pairs of the copy workload's shape in a pool of
    2 x pairs blocks, set up once; ``run()`` times the oracle's block copy
    (single-threaded C, plus the copies of the caches its Python wrapper
    returns, which grow with the pool)."""

    def __init__(self, pairs):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.pairs = pairs
        g = np.random.default_rng(7)
        nb = 2 * pairs
        self.kc = g.integers(0, 1 << 16, (nb, 8, 16, 128), dtype=np.uint16)
        self.vc = g.integers(0, 1 << 16, (nb, 8, 16, 128), dtype=np.uint16)
        perm = g.permutation(nb).astype(np.int32)
        self.src, self.dst = perm[:pairs], perm[pairs:]
        oracle.copy_blocks(self.kc[:4], self.vc[:4], self.src[:0], self.dst[:0])  # load the library
        self.sample = (f"{pairs} pairs in a pool of {nb} blocks of the same shape "
                       "(oracle_copy_blocks, one thread, with the wrapper's copies of both caches)")

    def run(self):
        t0 = time.perf_counter()
        self.oracle.copy_blocks(self.kc, self.vc, self.src, self.dst)
        sec = time.perf_counter() - t0
        moved = 2 * self.pairs * 2 * 8 * 16 * 128 * 2
        return moved / sec / 1e9, sec


def cow_cpu_baseline(pairs=COW_PAIRS):
    """The oracle's block copy on a sample of ``pairs`` pairs."""
    smp = CowOracleSample(pairs)
    v, sec = smp.run()
    return v, sec, smp.sample


def run_cow(args, rank, world, local_rank):
    """Copy-on-write block copies (the f2 row): one step = one pa_copy_blocks
    call over COW_PAIRS pairs; bytes read + written per second against the
    measured HBM copy bandwidth."""
    from paged_kv_cache_blocks_gb300 import build as pb_build
    pb_build.build()
    from paged_kv_cache_blocks_gb300 import binding as pa
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    Hkv, D, dt = 8, 128, torch.bfloat16
    g = torch.Generator(device=dev)
    g.manual_seed(5000 + rank)
    kc = torch.randn((COW_POOL, Hkv, 16, D), generator=g, device=dev).to(dt)
    vc = torch.randn((COW_POOL, Hkv, 16, D), generator=g, device=dev).to(dt)
    src, dst = cow_pairs(rank)
    src_d, dst_d = src.to(dev), dst.to(dev)
    per_pair = 2 * Hkv * 16 * D * 2                 # K and V of one block, bytes
    moved = 2 * per_pair * COW_PAIRS                # read + written per step
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        pa.pa_copy_blocks(kc, vc, src_d, dst_d)
    torch.cuda.synchronize()
    # the copy is idempotent once done: check it against the sources
    if not (torch.equal(kc[dst.long()], kc[src.long()]) and torch.equal(vc[dst.long()], vc[src.long()])):
        raise RuntimeError("pa_copy_blocks: destinations differ from sources after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    sampler = ClockSampler(gpu_identity(local_rank)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_host0 = time.time()
    start.record(stream)
    for a, z in ev:
        a.record(stream)
        pa.pa_copy_blocks(kc, vc, src_d, dst_d)
        z.record(stream)
    stop.record(stream)
    barrier()
    t_host1 = time.time()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    ms_step = reduce_max(start.elapsed_time(stop) / args.steps, dist, dev)
    times = sorted(a.elapsed_time(z) for a, z in ev)
    kern_ms = statistics.fmean(times)
    peak_gbs, peak_src = measured_peaks()
    e2e = None
    if not args.no_e2e:
        # through the public API: pair lists up from pinned host memory, the
        # copy, one destination block of K read back as the step's result
        src_h, dst_h = src.pin_memory(), dst.pin_memory()
        res_h = torch.empty((Hkv, 16, D), dtype=dt).pin_memory()
        probe = int(dst[0])
        steps = max(1, min(args.steps, args.e2e_steps))
        for _ in range(3):
            src_d.copy_(src_h, non_blocking=True)
            dst_d.copy_(dst_h, non_blocking=True)
            pa.pa_copy_blocks(kc, vc, src_d, dst_d)
            res_h.copy_(kc[probe], non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(steps):
            src_d.copy_(src_h, non_blocking=True)
            dst_d.copy_(dst_h, non_blocking=True)
            pa.pa_copy_blocks(kc, vc, src_d, dst_d)
            res_h.copy_(kc[probe], non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        sec = reduce_max((time.perf_counter() - t0) / steps, dist, dev)
        e2e = {"value": job_throughput(moved, world, sec) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": 2 * 4 * COW_PAIRS, "d2h_bytes_per_step": Hkv * 16 * D * 2,
               "steps": steps, "ms_per_step": sec * 1e3,
               "path": "per step: H2D (pinned) source and destination ids -> pa_copy_blocks -> "
                       "D2H of one copied K block; synchronised after the last step"}

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, sec, sample = cow_cpu_baseline()
        cpu = {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "seconds": sec,
               "sample": sample}
    line = {
        "metric": COW_METRIC, "value": job_throughput(moved, world, ms_step * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCR["cow"], "pairs": COW_PAIRS, "pool_blocks": COW_POOL,
                   "bytes_per_step": moved,
                   "l2": f"{moved / 2**20:.0f} MB read + written per step vs 129 MB L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": moved / (kern_ms * 1e-3) / 1e9,
                     "peak": peak_gbs, "unit": "GB/s",
                     "frac": moved / (kern_ms * 1e-3) / 1e9 / peak_gbs,
                     "traffic": load_traffic("cow", "auto"),
                     "traffic_gbs": (load_traffic("cow", "auto") / (kern_ms * 1e-3) / 1e9
                                     if load_traffic("cow", "auto") else None),
                     "kernel": "copy_blocks_kernel",
                     "kernel_ms": kern_ms,
                     "kernel_ms_p10_p50_p90": [times[len(times) // 10], times[len(times) // 2],
                                               times[(9 * len(times)) // 10]],
                     "algorithmic_bytes": moved,
                     "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": sampler.summary(t_host0, t_host1) if sampler else None,
    }
    if cpu is not None:
        cpu["cpu_model"] = cpu_model()
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


def run_reference_cow(args, rank, world):
    """The oracle's block copy as the reference arm of the copy workload:
    each step the same sample of pairs, sized from a 64-pair probe so that
    the whole run fits ``--ref-seconds``."""
    if rank != 0:
        return 0
    _, t64 = CowOracleSample(64).run()
    pairs = int(max(16, min(COW_PAIRS, 64 * ref_step_budget(args) // max(t64, 1e-6))))
    smp = CowOracleSample(pairs)
    vals = [smp.run() for _ in range(args.warmup + args.steps)][args.warmup:]
    v = statistics.fmean(x for x, _ in vals)
    sec = statistics.fmean(t for _, t in vals)
    line = {"impl": "reference", "metric": COW_METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": DESCR["cow"], "parallelism": "oracle, one thread",
                                            "sample": smp.sample},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": smp.sample, "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    from paged_kv_cache_blocks_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    threads = len(os.sched_getaffinity(0))
    lens_all = np.asarray(W.workload_lengths(args.workload, 0))
    # each step the same sample of the workload's sequences, as large as the
    # per-step budget allows: probe the smallest sample that keeps the
    # short/long mix, scale it up, or fall back to short sequences alone
    budget = ref_step_budget(args)
    mixed = bool((lens_all > 10 * np.median(lens_all)).any())
    rows = oracle_sample_rows(lens_all, 1)
    t1, _, _ = time_oracle(args.workload, rows, threads)
    if t1 <= budget:
        rows = oracle_sample_rows(lens_all, int(min(26 if mixed else len(lens_all), budget // t1)))
    elif mixed:
        short_rows = np.flatnonzero(lens_all <= 10 * np.median(lens_all))
        ts, _, _ = time_oracle(args.workload, short_rows[:1], threads)
        rows = short_rows[:int(max(1, min(len(short_rows), budget // max(ts, 1e-6))))]
    import oracle as O
    b = W.make_batch(args.workload, seed=0, poison=False,
                     lens_override=np.asarray(lens_all)[rows].tolist())
    kc, vc = W.place_new_tokens(b, 0)
    q = b.layers[0].q.numpy().view(np.uint16)
    kc, vc = kc.numpy().view(np.uint16), vc.numpy().view(np.uint16)
    for _ in range(args.warmup):
        O.decode(q, kc, vc, b.block_tables, b.seq_lens, w.scale, w.dtype, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.decode(q, kc, vc, b.block_tables, b.seq_lens, w.scale, w.dtype, threads=threads)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    kvb = logical_kv_bytes(b.seq_lens, w.num_kv_heads, w.head_dim)
    val = kvb / dt / 1e9
    sample = (f"{len(b.seq_lens)} of the {len(lens_all)} sequences of the workload "
              f"({int(np.sum(b.seq_lens))} tokens) per step, fp64 oracle, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": DESCR.get(args.workload, args.workload),
                                            "sample": sample},
            "seqs_steps_per_s": len(b.seq_lens) / dt,
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm

def run_pa(args, rank, world, local_rank):
    from paged_kv_cache_blocks_gb300 import build as pb
    pb.build()
    from paged_kv_cache_blocks_gb300 import binding as pa
    from paged_kv_cache_blocks_gb300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = W.WORKLOADS[args.workload]
    b = W.make_batch(args.workload, seed=rank, poison=False, device="cuda", num_layers=args.layers)
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    layers = [(Lr.q.view(dt), Lr.k_cache.view(dt), Lr.v_cache.view(dt), Lr.new_k.view(dt),
               Lr.new_v.view(dt)) for Lr in b.layers]
    kv_elem = 2
    if args.fp8:   # E4M3 caches (K token-major, V dimension-major), per-KV-head scales
        kv_elem = 1
        k_sc = torch.tensor([0.02 + 0.005 * h for h in range(w.num_kv_heads)], device=dev)
        v_sc = torch.tensor([0.03 + 0.004 * h for h in range(w.num_kv_heads)], device=dev)
        q8 = []
        for (q, kc, vc, nk, nv) in layers:
            k8 = (kc.float() / k_sc.view(1, -1, 1, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
            v8 = (vc.float() / v_sc.view(1, -1, 1, 1)).to(torch.float8_e4m3fn).view(torch.uint8) \
                .transpose(2, 3).contiguous()
            q8.append((q, k8, v8, nk, nv))
        layers = q8
        for Lr in b.layers:
            Lr.k_cache = Lr.v_cache = None
        torch.cuda.empty_cache()
    nl = len(layers)
    tab = torch.from_numpy(b.block_tables).to(dev)
    lens = torch.from_numpy(b.seq_lens).to(dev)
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    msl = int(b.seq_lens.max())
    grouped = args.grouped and any(m > 1 and p > 0 for m, p in b.groups)
    if grouped:
        goff, gpre = (torch.from_numpy(x).to(dev) for x in b.group_arrays())
        ws = torch.empty(pa.pa_decode_grouped_workspace_bytes(B, Hq, D, msl), dtype=torch.uint8,
                         device=dev)
    else:
        ws = torch.empty(pa.pa_decode_workspace_bytes(B, Hq, D, msl), dtype=torch.uint8, device=dev)
    out = torch.empty_like(layers[0][0])
    variant = VARIANTS[args.variant]
    stream = torch.cuda.current_stream()

    def step(evs=None):
        for li, (q, kc, vc, nk, nv) in enumerate(layers):
            ev = evs[li] if evs else None
            rp = li > 0   # the later layers of a step reuse the first layer's plan
            if args.fp8:
                pa.pa_cache_write_fp8(nk, nv, slots, k_sc, v_sc, kc, vc)
                pa.pa_decode_fp8(q, kc, vc, k_sc, v_sc, tab, lens, w.scale, max_seq_len=msl,
                                 out=out, workspace=ws, events=ev, reuse_plan=rp)
                continue
            pa.pa_cache_write(nk, nv, slots, kc, vc)
            if grouped:
                pa.pa_decode_grouped(q, kc, vc, tab, lens, w.scale, goff, gpre, max_seq_len=msl,
                                     out=out, workspace=ws, variant=variant, events=ev,
                                     reuse_plan=rp)
            else:
                pa.pa_decode(q, kc, vc, tab, lens, w.scale, max_seq_len=msl, out=out, workspace=ws,
                             variant=variant, events=ev, reuse_plan=rp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bits = pa.pa_decode_check(ws)
    if bits:
        raise RuntimeError(f"device error bits {bits} during warm-up")

    ev_pairs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(nl)] for _ in range(args.steps)]
    for row in ev_pairs:   # torch creates the CUDA event on its first record
        for a, z in row:
            a.record(stream)
            z.record(stream)
    sampler = ClockSampler(gpu_identity(local_rank)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_host0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step()
    stop.record(stream)
    barrier()
    t_host1 = time.time()
    # the attention kernel alone: the same steps again with events around each
    # of its launches (kept out of the step timing above: an event recorded
    # between two kernels keeps the second from starting during the first's tail)
    for i in range(args.steps):
        step(ev_pairs[i])
    barrier()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    ms_total = start.elapsed_time(stop)
    kern_ms = [a.elapsed_time(z) for row in ev_pairs for a, z in row]
    ms_step = reduce_max(ms_total / args.steps, dist, dev)

    kvb = logical_kv_bytes(b.seq_lens, Hkv, D, elem=kv_elem) * nl
    kv_gbs = job_throughput(kvb, world, ms_step * 1e-3) / 1e9
    part_tokens = int(ws[24:28].view(torch.int32).item())   # chosen by the prep kernel
    starts = None
    if grouped:   # the attention kernel covers each member's tokens past the shared prefix
        starts = np.repeat([p for _, p in b.groups], [m for m, _ in b.groups])
    alg = algorithmic_bytes(b.seq_lens, Hq, Hkv, D, part_tokens=part_tokens, kv_elem=kv_elem,
                            starts=starts)
    kern_avg = statistics.fmean(kern_ms)
    kq = np.percentile(np.asarray(kern_ms), [10, 50, 90]) if kern_ms else [float("nan")] * 3
    peak, peak_kind = measured_peaks()
    achieved = alg / (kern_avg * 1e-3) / 1e9

    # ---- the same step replayed from a CUDA graph (launch gaps removed) ---------
    graph = None
    if args.graph:
        graph = time_graph(step, args.steps, args.warmup, stream, barrier, dist, dev, kvb, world)

    # ---- end to end through the public API, host buffers -------------------------
    e2e = run_e2e(args, pa, W, b, w, dt, dev, variant, barrier, world, dist, grouped,
                  (k_sc, v_sc) if args.fp8 else None) \
        if not args.no_e2e else None

    # ---- every decode config of the workload table, measured the same way ---------
    per_config = None
    if args.per_config and world == 1 and not args.fp8 and not grouped:
        per_config = {}
        for name in PER_CONFIG:
            try:
                per_config[name] = measure_config(pa, W, name, args.steps, args.warmup, dev,
                                                  measured_peaks()[0],
                                                  with_oracle=not args.no_cpu_baseline)
            except Exception as ex:   # report, do not hide
                per_config[name] = {"error": repr(ex)}

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        try:
            cpu = cpu_baseline(args.workload)
        except Exception as ex:  # report, do not hide
            cpu = {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle",
                   "sample": f"failed: {ex!r}"}
    traffic = load_traffic(args.workload, "fp8" if args.fp8 else
                           ("grouped" if grouped else args.variant))
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    line = {
        "metric": METRIC, "value": kv_gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("fp8-e4m3 KV, " if args.fp8 else "") + ("bf16" if w.dtype == "bf16" else "f16"),
        "data": "synthetic",
        "config": {"workload": DESCR.get(args.workload, args.workload),
                   "num_seqs": B, "layers": nl, "kv_tokens": int(b.seq_lens.sum()),
                   "logical_kv_bytes_per_step": kvb,
                   "unique_kv_bytes_per_step": b.unique_kv_bytes() * nl * kv_elem // 2,
                   "l2": f"inputs larger than L2: {kvb / 1e9:.2f} GB of KV per step vs 129 MB L2; "
                         "no flush",
                   "step": f"{nl} x (pa_cache_write of one new token per sequence + pa_decode)"
                           + (" (layers after the first reuse its partition plan)" if nl > 1 else ""),
                   "variant": args.variant, "partition_tokens": part_tokens,
                   "shared_prefix": "pa_decode_grouped (prefix read once per group and KV head)"
                                    if grouped else "none (pa_decode)",
                   "parallelism": f"replicas x{world}"},
        "seqs_steps_per_s": job_throughput(B, world, ms_step * 1e-3),
        "hbm_frac_step": (kvb / (ms_step * 1e-3) / 1e9) / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic_gbs": traffic / (kern_avg * 1e-3) / 1e9 if traffic else None,
                     "traffic_frac": traffic / (kern_avg * 1e-3) / 1e9 / peak if traffic else None,
                     "kernel": "attend_fp8_kernel" if args.fp8 else "attend_kernel", "kernel_ms": kern_avg,
                     "kernel_ms_p10_p50_p90": [float(x) for x in kq],
                     "algorithmic_bytes": alg, "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": e2e,
        "graph": graph,
        # per layer: cache write, attention, merge (+ prefix kernel when grouped);
        # one prep per step (the later layers reuse its plan)
        "gpu_launches": ((3 + int(grouped)) * nl + 1) * args.steps,
        "clocks": clocks,
    }
    if per_config is not None:
        line["per_config"] = per_config
    if cpu is not None:
        cpu["cpu_model"] = cpu_model()
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- every decode config

PER_CONFIG = ("tiny", "llama8b", "llama70b", "long", "fullstep")
L2_BYTES = 129 * 1000 * 1000          # GB300 L2, for the flush decision
NOMINAL_HBM_GBS = 7900.0              # GB300 HBM3e nominal bandwidth (context only)


def cache_write_bytes(T, hkv, d, elem=2):
    """One cache write: k and v rows read, the same bytes written."""
    return 2 * 2 * T * hkv * d * elem


def oracle_config_times(name, b):
    """The fp64 oracle on one layer of the config's batch (its own host
    cores, all of them), and on one thread over its first two sequences."""
    import oracle
    oracle.build()
    from paged_kv_cache_blocks_gb300 import workloads as W
    w = b.workload
    kc, vc = W.place_new_tokens(b, 0)
    kc, vc = kc.cpu().numpy().view(np.uint16), vc.cpu().numpy().view(np.uint16)
    q = b.layers[0].q.cpu().numpy().view(np.uint16)
    threads = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    oracle.decode(q, kc, vc, b.block_tables, b.seq_lens, w.scale, w.dtype, threads=threads)
    t_all = time.perf_counter() - t0
    n1 = min(2, len(b.seq_lens))
    t0 = time.perf_counter()
    oracle.decode(q[:n1], kc, vc, b.block_tables[:n1], b.seq_lens[:n1], w.scale, w.dtype, threads=1)
    t_one = time.perf_counter() - t0
    tok_all, tok_one = int(b.seq_lens.sum()), int(b.seq_lens[:n1].sum())
    return {"oracle_layer_s": t_all, "oracle_threads": threads,
            "oracle_kv_gbs": logical_kv_bytes(b.seq_lens, w.num_kv_heads, w.head_dim) / t_all / 1e9,
            "oracle_1thread_layer_s_est": t_one * tok_all / max(tok_one, 1),
            "oracle_1thread_sample": f"{n1} sequences ({tok_one} tokens), scaled by tokens"}


def measure_config(pa, W, name, steps, warmup, dev, peak, with_oracle=True):
    """One decode config measured the way the headline is: a step = per
    layer pa_cache_write of every sequence's new token + pa_decode (layers
    after the first reuse the first layer's plan), CUDA events around each
    step and around each attention launch.  Configs whose KV is under 4x the
    L2 size get the L2 flushed (a 256 MB write, then a 256 MB read) before
    every step, outside the timed region; the others stream more than L2
    holds anyway."""
    w = W.WORKLOADS[name]
    b = W.make_batch(name, seed=0, poison=False, device="cuda")
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    layers = [(Lr.q.view(dt), Lr.k_cache.view(dt), Lr.v_cache.view(dt), Lr.new_k.view(dt),
               Lr.new_v.view(dt)) for Lr in b.layers]
    nl = len(layers)
    tab = torch.from_numpy(b.block_tables).to(dev)
    lens = torch.from_numpy(b.seq_lens).to(dev)
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    msl = int(b.seq_lens.max())
    ws = torch.empty(pa.pa_decode_workspace_bytes(B, Hq, D, msl), dtype=torch.uint8, device=dev)
    out = torch.empty_like(layers[0][0])
    kvb = logical_kv_bytes(b.seq_lens, Hkv, D) * nl
    flush = kvb < 4 * L2_BYTES
    if flush:
        flush_w = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
        flush_r = torch.zeros(64 * 2 ** 20, dtype=torch.int32, device=dev)

    def l2_flush():
        # write a buffer twice the L2 size, then read another one: the dirty
        # lines the write leaves are written back during the read, so the
        # timed step starts with an L2 of clean, unrelated lines
        flush_w.zero_()
        torch.max(flush_r)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        for li, (q, kc, vc, nk, nv) in enumerate(layers):
            pa.pa_cache_write(nk, nv, slots, kc, vc)
            pa.pa_decode(q, kc, vc, tab, lens, w.scale, max_seq_len=msl, out=out, workspace=ws,
                         events=evs[li] if evs else None, reuse_plan=li > 0)

    for _ in range(warmup):
        if flush:
            l2_flush()
        step()
    torch.cuda.synchronize()
    if pa.pa_decode_check(ws):
        raise RuntimeError(f"{name}: device error bits during warm-up")
    mk = lambda: torch.cuda.Event(enable_timing=True)
    st_ev = [(mk(), mk()) for _ in range(steps)]
    k_ev = [[(mk(), mk()) for _ in range(nl)] for _ in range(steps)]
    for row in k_ev:
        for a, z in row:
            a.record(stream)
            z.record(stream)
    torch.cuda.synchronize()
    # steps timed as a whole (events only around each step), then the same
    # steps with events around each attention launch for the kernel's time
    for i in range(steps):
        if flush:
            l2_flush()
        st_ev[i][0].record(stream)
        step()
        st_ev[i][1].record(stream)
    for i in range(steps):
        if flush:
            l2_flush()
        step(k_ev[i])
    torch.cuda.synchronize()
    step_ms = statistics.fmean(a.elapsed_time(z) for a, z in st_ev)
    kern_ms = statistics.fmean(a.elapsed_time(z) for row in k_ev for a, z in row)
    part_tokens = int(ws[24:28].view(torch.int32).item())
    alg = algorithmic_bytes(b.seq_lens, Hq, Hkv, D, part_tokens=part_tokens)
    step_alg = nl * (alg + cache_write_bytes(B, Hkv, D))
    r = {"workload": DESCR[name], "num_seqs": B, "layers": nl,
         "kv_tokens_per_layer": int(b.seq_lens.sum()), "logical_kv_bytes_per_step": kvb,
         "ms_per_step": step_ms, "us_per_step": step_ms * 1e3,
         "kv_gbs": kvb / (step_ms * 1e-3) / 1e9,
         "seqs_steps_per_s": B / (step_ms * 1e-3),
         "attend_us_per_launch": kern_ms * 1e3,
         "attend_frac": alg / (kern_ms * 1e-3) / 1e9 / peak,
         "step_alg_frac": step_alg / (step_ms * 1e-3) / 1e9 / peak,
         "partition_tokens": part_tokens,
         "l2": "flushed before every step (256 MB written, then 256 MB read; not timed)" if flush
               else f"not flushed: {kvb / 1e9:.2f} GB of KV per step vs 129 MB L2"}
    if name == "tiny":   # latency-bound: report time only
        for k in ("kv_gbs", "attend_frac", "step_alg_frac"):
            r.pop(k)
    if name == "fullstep":
        goff, gpre = (torch.from_numpy(x).to(dev) for x in b.group_arrays())
        gws = torch.empty(pa.pa_decode_grouped_workspace_bytes(B, Hq, D, msl), dtype=torch.uint8,
                          device=dev)

        def gstep():
            for li, (q, kc, vc, nk, nv) in enumerate(layers):
                pa.pa_cache_write(nk, nv, slots, kc, vc)
                pa.pa_decode_grouped(q, kc, vc, tab, lens, w.scale, goff, gpre, max_seq_len=msl,
                                     out=out, workspace=gws, reuse_plan=li > 0)
        for _ in range(warmup):
            gstep()
        a, z = mk(), mk()
        a.record(stream)
        for _ in range(steps):
            gstep()
        z.record(stream)
        torch.cuda.synchronize()
        r["grouped_ms_per_step"] = a.elapsed_time(z) / steps
        r["unique_kv_bytes_per_step"] = b.unique_kv_bytes() * nl
    if with_oracle:
        r.update(oracle_config_times(name, b))
        if nl > 1:
            r["oracle_note"] = f"one layer timed; a {nl}-layer step takes {nl}x"
    del layers, b
    torch.cuda.empty_cache()
    return r


def time_graph(step, steps, warmup, stream, barrier, dist, dev, units, world):
    """Capture one step in a CUDA graph and time `steps` replays (the library
    calls neither synchronise nor allocate, so the whole step is capturable).
    Returns the step time and the throughput of `units` bytes per step."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(max(warmup, 3)):
        g.replay()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    a.record(stream)
    for _ in range(steps):
        g.replay()
    z.record(stream)
    barrier()
    ms = reduce_max(a.elapsed_time(z) / steps, dist, dev)
    return {"ms_per_step": ms, "value": job_throughput(units, world, ms * 1e-3) / 1e9,
            "unit": "GB/s", "how": "one step captured in a CUDA graph, replayed back to back"}


# dram__bytes_read.sum + dram__bytes_write.sum of one attention launch, from
# the ncu captures summarised in profiles/ (file named below), keyed by the
# hash of the kernel sources they were taken on: a changed kernel reports null.
TRAFFIC = {
    ("llama70b", "auto"): {"bytes": 3773.76e6 + 9.35e6, "kernel_src": "e0b3982bd76effc8",
                           "profile": "profiles/attend_kernel_llama70b_dram.md"},
    ("llama70b", "mma"): {"bytes": 3773.76e6 + 9.35e6, "kernel_src": "e0b3982bd76effc8",
                          "profile": "profiles/attend_kernel_llama70b_dram.md"},
    ("llama70b", "fp8"): {"bytes": 1889.38e6 + 3.37e6, "kernel_src": "e0b3982bd76effc8",
                          "profile": "profiles/decode_step_llama70b_fp8_launches.md"},
    ("fullstep", "auto"): {"bytes": 1978.47e6 + 4.28e6, "kernel_src": "e0b3982bd76effc8",
                           "profile": "profiles/attend_kernel_fullstep_shared_prefix_l2.md"},
    ("fullstep", "grouped"): {"bytes": 1937.99e6 + 3.73e6, "kernel_src": "e0b3982bd76effc8",
                              "profile": "profiles/attend_kernel_fullstep_shared_prefix_l2.md"},
    ("cow", "auto"): {"bytes": 268.53e6 + 216.54e6, "kernel_src": "52affb2a945dc192",
                      "profile": "profiles/copy_blocks_kernel_cow.md"},
    # the 8 prefill launches of one step (iterations 1..8), summed
    ("chunked", "auto"): {"bytes": 1285.57e6 + 286.94e6, "kernel_src": "3609587c3737d282",
                          "profile": "profiles/prefill_tc_kernel_chunked.md"},
}


DECODE_SRC = ("pa_decode.cu", "pa_device.cuh")
PREFILL_SRC = ("pa_prefill.cu", "pa_device.cuh")
COPY_SRC = ("pa_cache_write.cu", "pa_device.cuh")


def kernel_src_hash(files=DECODE_SRC):
    """First 16 hex of the sha256 of the kernel sources with comments and
    whitespace removed, so that only a change of code invalidates counters."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_blocks_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def load_traffic(workload, variant):
    """DRAM bytes per attention launch (per step of 8 launches for the
    chunked prefill) from the ncu capture of this kernel build, or None when
    there is none (or the kernel changed since)."""
    ent = TRAFFIC.get((workload, variant))
    files = {"chunked": PREFILL_SRC, "cow": COPY_SRC}.get(workload, DECODE_SRC)
    if not ent or ent["kernel_src"] != kernel_src_hash(files):
        return None
    return ent["bytes"]


def run_e2e(args, pa, W, b, w, dt, dev, variant, barrier, world, dist, grouped=False,
            scales=None):
    """Same step through the public API from pinned host memory (E4M3 caches
    with ``args.fp8``; shared-prefix groups decoded by pa_decode_grouped when
    ``grouped``)."""
    import ctypes
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    nl = len(b.layers)
    steps = max(1, min(args.steps, args.e2e_steps))
    total = steps + args.warmup
    lens0 = b.seq_lens.astype(np.int64) - 1
    mb = int(((lens0 + total + 15) // 16).max())
    need = int(((lens0 + total + 15) // 16).sum())
    nb = max(b.num_blocks, int(math.ceil(need * 1.05)))
    order = np.random.default_rng(123).permutation(nb).astype(np.int32)
    alloc = pa.Allocator(nb, order)
    table_h = torch.full((B, mb), -1, dtype=torch.int32).pin_memory()
    lens_h = torch.zeros(B, dtype=torch.int32).pin_memory()
    scratch = np.empty(int(lens0.max()) + 1, np.int64)

    def append(i, sid, n):
        one = np.array([sid], np.int64)
        rc = pa.lib().pa_seq_append_slots(alloc._h, one.ctypes.data, 1, int(n), scratch.ctypes.data,
                                          None, None, 0, None, table_h[i:i + 1].numpy().ctypes.data,
                                          mb, lens_h[i:i + 1].numpy().ctypes.data)
        if rc != 0:
            raise RuntimeError(pa.lib().pa_last_error_string().decode())

    ids = np.zeros(B, np.int64)
    if w.name == "fullstep":   # groups share a prefix through fork (ref-counted blocks)
        per = B // W.PREFIX_GROUPS
        for gi in range(W.PREFIX_GROUPS):
            parent = alloc.seq_create()
            append(gi * per, parent, W.PREFIX_TOKENS)
            for i in range(gi * per, (gi + 1) * per):
                ids[i] = alloc.seq_fork(parent, W.PREFIX_TOKENS)
            alloc.seq_free(parent)
        rows, _ = alloc.block_table(ids.tolist(), mb)
        table_h.copy_(torch.tensor(rows, dtype=torch.int32))
        lens_h.fill_(W.PREFIX_TOKENS)
        for i in range(B):
            append(i, ids[i], lens0[i] - W.PREFIX_TOKENS)
    else:
        for i in range(B):  # the tokens already in the cache
            ids[i] = alloc.seq_create()
            if lens0[i] > 0:
                append(i, ids[i], lens0[i])
    ids_c = ids.ctypes.data_as(ctypes.c_void_p)
    g = torch.Generator().manual_seed(99)
    # step inputs in pinned host memory (q/k/v per layer; metadata rewritten by
    # the allocator every step) and the step's outputs, read back every step
    q_h = [torch.randn((B, Hq, D), generator=g).to(dt).pin_memory() for _ in range(nl)]
    k_h = [torch.randn((B, Hkv, D), generator=g).to(dt).pin_memory() for _ in range(nl)]
    v_h = [torch.randn((B, Hkv, D), generator=g).to(dt).pin_memory() for _ in range(nl)]
    out_h = [[torch.empty((B, Hq, D), dtype=dt).pin_memory() for _ in range(nl)] for _ in range(2)]
    slots_h = torch.empty(B, dtype=torch.int64).pin_memory()
    if args.fp8:   # K token-major, V dimension-major bytes
        caches = [(torch.zeros((nb, Hkv, 16, D), dtype=torch.uint8, device=dev),
                   torch.zeros((nb, Hkv, D, 16), dtype=torch.uint8, device=dev)) for _ in range(nl)]
        k_sc, v_sc = scales
    else:
        caches = [(torch.zeros((nb, Hkv, 16, D), dtype=dt, device=dev),
                   torch.zeros((nb, Hkv, 16, D), dtype=dt, device=dev)) for _ in range(nl)]
    meta_h = [slots_h, table_h, lens_h]
    if grouped:
        meta_h += [torch.from_numpy(x).pin_memory() for x in b.group_arrays()]
    msl = mb * 16

    # two device slots: step i uses slot i % 2, so that the copies of step i
    # overlap the compute of step i - 1
    class Slot:
        pass
    slots = []
    for _ in range(2):
        sl = Slot()
        sl.q = [torch.empty((B, Hq, D), dtype=dt, device=dev) for _ in range(nl)]
        sl.k = [torch.empty((B, Hkv, D), dtype=dt, device=dev) for _ in range(nl)]
        sl.v = [torch.empty((B, Hkv, D), dtype=dt, device=dev) for _ in range(nl)]
        sl.out = [torch.empty((B, Hq, D), dtype=dt, device=dev) for _ in range(nl)]
        sl.meta = [torch.empty_like(x, device=dev) for x in meta_h]
        sl.meta_copied = torch.cuda.Event()
        sl.inputs_ready = torch.cuda.Event()
        sl.comp_done = torch.cuda.Event()
        slots.append(sl)
    if grouped:
        ws = torch.empty(pa.pa_decode_grouped_workspace_bytes(B, Hq, D, msl), dtype=torch.uint8,
                         device=dev)
    else:
        ws = torch.empty(pa.pa_decode_workspace_bytes(B, Hq, D, msl), dtype=torch.uint8, device=dev)
    slots_np, table_np, lens_np = slots_h.numpy(), table_h.numpy(), lens_h.numpy()
    nbytes = lambda t: t.numel() * t.element_size()
    h2d = sum(nbytes(t) for t in q_h + k_h + v_h) + sum(nbytes(t) for t in meta_h)
    d2h = sum(nbytes(t) for t in out_h[0])
    kv_bytes = []
    compute = torch.cuda.current_stream()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    state = {"i": 0}

    def one_step():
        i = state["i"]
        sl = slots[i & 1]
        if i >= 1:   # the pinned metadata is free once the previous step's copy ran
            slots[(i - 1) & 1].meta_copied.synchronize()
        rc = pa.lib().pa_seq_append_slots(alloc._h, ids_c, B, 1, slots_np.ctypes.data, None, None,
                                          0, None, table_np.ctypes.data, mb, lens_np.ctypes.data)
        if rc != 0:
            raise RuntimeError(pa.lib().pa_last_error_string().decode())
        with torch.cuda.stream(h2d_stream):
            if i >= 2:   # this slot's buffers are free once step i - 2 computed
                h2d_stream.wait_event(sl.comp_done)
            for hx, dx in zip(meta_h, sl.meta):
                dx.copy_(hx, non_blocking=True)
            sl.meta_copied.record(h2d_stream)
            for li in range(nl):
                sl.q[li].copy_(q_h[li], non_blocking=True)
                sl.k[li].copy_(k_h[li], non_blocking=True)
                sl.v[li].copy_(v_h[li], non_blocking=True)
            sl.inputs_ready.record(h2d_stream)
        compute.wait_event(sl.inputs_ready)
        slots_d, table_d, lens_d = sl.meta[0], sl.meta[1], sl.meta[2]
        for li in range(nl):
            kc, vc = caches[li]
            rp = li > 0   # the later layers of a step reuse the first layer's plan
            if args.fp8:
                pa.pa_cache_write_fp8(sl.k[li], sl.v[li], slots_d, k_sc, v_sc, kc, vc)
                pa.pa_decode_fp8(sl.q[li], kc, vc, k_sc, v_sc, table_d, lens_d, w.scale,
                                 max_seq_len=msl, out=sl.out[li], workspace=ws, reuse_plan=rp)
            else:
                pa.pa_cache_write(sl.k[li], sl.v[li], slots_d, kc, vc)
                if grouped:
                    pa.pa_decode_grouped(sl.q[li], kc, vc, table_d, lens_d, w.scale, *sl.meta[3:5],
                                         max_seq_len=msl, out=sl.out[li], workspace=ws,
                                         variant=variant, reuse_plan=rp)
                else:
                    pa.pa_decode(sl.q[li], kc, vc, table_d, lens_d, w.scale, max_seq_len=msl,
                                 out=sl.out[li], workspace=ws, variant=variant, reuse_plan=rp)
        sl.comp_done.record(compute)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(sl.comp_done)
            for li in range(nl):
                out_h[i & 1][li].copy_(sl.out[li], non_blocking=True)
        kv_bytes.append(int(lens_np.astype(np.int64).sum()) * Hkv * D * 2 * (1 if args.fp8 else 2)
                        * nl)
        state["i"] = i + 1

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    kv_bytes.clear()
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    torch.cuda.synchronize()
    barrier()
    sec = reduce_max((time.perf_counter() - t0) / steps, dist, dev)
    alloc.close()
    return {"value": job_throughput(statistics.fmean(kv_bytes), world, sec) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": sec * 1e3,
            "path": "per step: host allocator append_slots -> H2D (pinned, copy stream) slots,table,lens"
                    + (",group offsets/prefixes" if grouped else "") + " and per layer q,k,v -> "
                    + ("pa_cache_write_fp8 -> pa_decode_fp8" if args.fp8 else
                       "pa_cache_write -> " + ("pa_decode_grouped" if grouped else "pa_decode"))
                    + " -> D2H out (second copy stream); two device slots let step i's copies "
                      "overlap step i-1's compute; synchronised after the last step"}


def run_reference_prefill(args, rank, world):
    """The oracle as the reference arm of the chunked workload: each step the
    same sample of query rows, sized from a four-row probe so that the whole
    run fits ``--ref-seconds``; FLOP/s scaled from the sample."""
    if rank != 0:
        return 0
    budget = ref_step_budget(args)
    smp = PrefillOracleSample()
    _, t4, _ = smp.run(4)
    if t4 / 4 > budget:
        # one row of the last piece (~28k visible keys) is over the budget:
        # take rows of the first piece (at most 3,750 visible keys) instead
        smp = PrefillOracleSample(iteration=1)
        _, t4, _ = smp.run(4)
    n_rows = int(max(1, min(smp.n, budget // max(t4 / 4, 1e-6))))
    for _ in range(args.warmup):
        smp.run(n_rows)
    vals, secs = [], []
    for _ in range(args.steps):
        v, sec, sample = smp.run(n_rows)
        vals.append(v)
        secs.append(sec)
    val = statistics.fmean(vals)
    threads = smp.threads
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.fmean(secs) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": DESCR["chunked"], "sample": sample},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama70b", choices=sorted(DESCR))
    ap.add_argument("--variant", default="auto", choices=sorted(VARIANTS))
    ap.add_argument("--impl", default="pa", choices=["pa", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--ref-seconds", type=float, default=REF_RUN_S,
                    help="--impl reference: oracle seconds for the whole run; each step's "
                         "sample of the workload is sized to fit")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="E4M3 KV caches: pa_cache_write_fp8 + pa_decode_fp8")
    ap.add_argument("--grouped", action="store_true",
                    help="decode shared-prefix groups with pa_decode_grouped (fullstep)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="skip timing the step replayed from a CUDA graph")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode only the first N layers of the workload (a smaller case to "
                         "profile; the line's config then names N layers)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip measuring every decode config after the headline")
    args = ap.parse_args()
    if args.fp8 and args.grouped:
        ap.error("--fp8 and --grouped do not combine (the shared-prefix kernel reads 16-bit caches)")
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if args.workload == "chunked":
            return run_reference_prefill(args, rank, world)
        if args.workload == "cow":
            return run_reference_cow(args, rank, world)
        return run_reference(args, rank, world)
    if args.workload == "chunked":
        return run_prefill(args, rank, world, local_rank)
    if args.workload == "cow":
        return run_cow(args, rank, world, local_rank)
    return run_pa(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
