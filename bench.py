"""Benchmark of the two-tier sparse-attention decode step on GB300.

Default workload: decode, batch 64, 131072 tokens per sequence at compression
ratio 1 (131072 latents, 16384 blocks of 8; the candidate stage keeps 2048
blocks), MXFP8 index keys, bf16 latents, top-512 plus a 128-position window.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one whole decode step: pooling of each sequence's newest block,
block scores + top-2048 blocks, token scores + top-512 latents, and attention,
for every query of the batch. Inputs (caches and queries) are resident in HBM
when the timed region starts; the L2 is flushed (a 512 MiB write, then a
256 MiB read pass) before every timed step, outside its events. The step is
captured once in a CUDA graph and each timed step is one replay (the
stream-launched figure is reported beside it). `value` is queries/s over the
whole job.
`e2e` repeats the step through the C ABI with host buffers: each step copies
its queries in from pinned host memory (q, q_idx and w in one packed copy) and
its outputs back (out and lse in one copy).
The reference arm times the CPU oracle on the host cores on a bounded sample.
Multi-GPU: one process per GPU (torchrun); decode shards by sequence, so each
rank runs its own batch with no collective (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode queries/s at 128K ctx; achieved HBM GB/s vs roofline"
PREFILL_METRIC = ("sparse-attn prefill queries/s (4096 queries on 64K context); achieved bf16 "
                  "TFLOP/s vs roofline")
PREFILL_CPU_SAMPLE = 512  # oracle queries timed for a prefill chunk's CPU figure
MULTI_METRIC = ("sparse-attn multi-query decode queries/s at 128K ctx (5 queries a sequence); "
                "achieved HBM GB/s vs roofline")
DEFAULT_WORKLOAD = "decode_b64_t131072_r1_mxfp8"
PREFILL_WORKLOAD = "prefill_q4096_ctx65536_r2_bf16"
L2_FLUSH_BYTES = 512 << 20
L2_READ_BYTES = 256 << 20


class L2Flush:
    """Evicts the L2 (129 MB) between timed steps. A write of 512 MiB alone
    leaves the L2 full of dirty lines, which the step's first large read then
    has to write back to HBM while it streams; a read-only pass over another
    256 MiB after the write cleans them out before the step starts."""

    DESCRIPTION = "flushed before every timed step (512 MiB write, then a 256 MiB read pass)"

    def __init__(self, dev):
        import torch

        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_READ_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--batch", type=int, default=0,
                   help="override the workload's batch (smaller cases for profiling)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true",
                   help="skip the prefill chunk that the default decode run measures after "
                        "its own steps (reported under extra.prefill)")
    p.add_argument("--cpu-sample", type=int, default=0,
                   help="sequences (decode) or queries (prefill) in the CPU-oracle sample (0: automatic)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank runs its own batch (weak scaling, no collective on the data
    path): its inputs come from its own seed."""
    return base_seed + 1000 * rank


def reduce_max(values, device):
    """Element-wise maximum of per-rank values over all ranks (the slowest
    rank's time sets the job's); the values unchanged for a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's units per step over the slowest
    rank's step time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def sustained_bf16_peak():
    """The bf16 GEMM rate measured over seconds under the power cap (for a
    kernel timed inside a long step), or None when it was not measured."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clocks, power and throttle reasons with single-shot
    nvidia-smi queries from a background thread (about every 100 ms) while the
    timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.stop = threading.Event()
        self.t = None

    def _run(self):
        while not self.stop.is_set():
            try:
                out = subprocess.run(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                     "--format=csv,noheader,nounits"],
                    capture_output=True, text=True, timeout=5).stdout
                self.lines.extend(x.strip() for x in out.splitlines() if x.strip())
            except Exception:
                pass
            self.stop.wait(0.1)

    def __enter__(self):
        if shutil.which("nvidia-smi"):
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.t is not None:
            self.t.join(timeout=10)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def cpu_oracle_rate(workload: str, n_seq: int, steps: int = 1):
    """Times the oracle, as it stands, on n_seq sequences of the workload's shape.
    Returns (queries/s, seconds per step, threads, sample description)."""
    import oracle as O
    import synth
    spec = dict(synth.WORKLOADS[workload])
    assert spec.pop("kind") == "decode"
    inp = synth.decode_inputs([spec["T"]] * n_seq, spec["ratio"], spec["key_fmt"], spec["seed"],
                              kv_fmt=spec.get("kv_fmt", "bf16"))
    cfg = O.StepConfig(ratio=spec["ratio"])
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        for b in range(n_seq):
            O.decode_sequence(cfg, inp, b)
        times.append(time.perf_counter() - t0)
    threads = int(os.environ.get("OMP_NUM_THREADS", "0")) or os.cpu_count() or 1
    sample = (f"{n_seq} sequence(s) of the workload ({spec['T']} tokens, ratio {spec['ratio']}, "
              f"{spec['key_fmt']} keys); the oracle pools each sequence's keys as part of its step")
    t = float(np.median(times))
    return n_seq / t, t, threads, sample


def cpu_oracle_prefill_rate(workload: str, n_sample: int, steps: int = 1):
    """Times the oracle, as it stands, on n_sample queries spread evenly over the
    workload's prefill chunk. The complete-block keys are built once outside the
    timed region, as the GPU step takes them from its cache; each query pools its
    own partly visible block. Returns (queries/s, seconds per step, threads,
    sample description)."""
    import oracle as O
    import synth
    spec = dict(synth.WORKLOADS[workload])
    assert spec.pop("kind") == "prefill"
    n_q, ctx, ratio, fmt = spec["n_q"], spec["ctx"], spec["ratio"], spec["key_fmt"]
    inp = synth.prefill_inputs(n_q, ctx, ratio, fmt, spec["seed"])
    cfg = O.StepConfig(ratio=ratio)
    kv, pooled, _ = O.prefill_caches(cfg, inp)
    picks = np.unique(np.linspace(0, n_q - 1, max(1, min(n_sample, n_q))).round().astype(int))
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        for i in picks:
            O.prefill_query(cfg, inp, int(i), kv, pooled)
        times.append(time.perf_counter() - t0)
    threads = int(os.environ.get("OMP_NUM_THREADS", "0")) or os.cpu_count() or 1
    sample = (f"{len(picks)} of the chunk's {n_q} queries, evenly spaced (context {ctx}, ratio "
              f"{ratio}, {fmt} keys); the complete-block keys are built once, outside the "
              "timed region")
    t = float(np.median(times))
    return len(picks) / t, t, threads, sample


def cpu_oracle_multi_rate(workload: str, n_seq: int, steps: int = 1):
    """Times the oracle, as it stands, on n_seq sequences of a multi-query
    workload (all of each sequence's queries, its block keys built inside the
    timed region as the decode leg does). Returns (queries/s, seconds per step,
    threads, sample description)."""
    import oracle as O
    import synth
    spec = dict(synth.WORKLOADS[workload])
    assert spec.pop("kind") == "multi"
    m = synth.multi_inputs([spec["T"]] * n_seq, spec["n_q"], spec["ratio"], spec["key_fmt"],
                           spec["seed"])
    cfg = O.StepConfig(ratio=spec["ratio"])
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        for b in range(n_seq):
            view = synth.multi_as_prefill(m, b)
            kv, pooled, _ = O.prefill_caches(cfg, view)
            for i in range(m.n_q):
                O.prefill_query(cfg, view, i, kv, pooled)
        times.append(time.perf_counter() - t0)
    threads = int(os.environ.get("OMP_NUM_THREADS", "0")) or os.cpu_count() or 1
    sample = (f"{n_seq} sequence(s) x {m.n_q} queries of the workload ({spec['T']} tokens, ratio "
              f"{spec['ratio']}, {spec['key_fmt']} keys); each sequence's block keys are built "
              "in the timed region")
    t = float(np.median(times))
    return n_seq * m.n_q / t, t, threads, sample


THREADS_NOTE = ("the oracle's loops run in one Python thread; numpy's BLAS calls inside them may "
                "use up to `cores` threads")


def cpu_oracle_one_thread(workload: str, n_seq: int):
    """The decode oracle timed again in a child process whose BLAS and OpenMP
    are held to one thread (environment set before numpy loads). Returns
    {"value", "unit", "threads": 1, "sample"} or None if the child failed."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_oracle_rate(%r, %d)))" % (ROOT, workload, n_seq))
    try:
        p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=900)
        qps, _, _, sample = json.loads(p.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return {"value": qps, "unit": "queries/s", "threads": 1, "sample": sample}


def auto_cpu_sample(workload: str) -> int:
    import synth
    T = synth.WORKLOADS[workload]["T"]
    return max(1, min(16, int(2 ** 21 // max(T, 1))))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth
    spec = synth.WORKLOADS[args.workload]
    if spec["kind"] == "multi":
        n = args.cpu_sample or 2
        for _ in range(args.warmup):
            cpu_oracle_multi_rate(args.workload, n)
        qps, t, threads, sample = cpu_oracle_multi_rate(args.workload, n, steps=max(1, args.steps))
        line = {
            "impl": "reference", "metric": MULTI_METRIC, "value": qps, "unit": "queries/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": spec["B"], "queries_per_seq": spec["n_q"],
                       "tokens": spec["T"], "ratio": spec["ratio"], "key_fmt": spec["key_fmt"]},
            "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    if spec["kind"] == "prefill":
        n = args.cpu_sample or PREFILL_CPU_SAMPLE
        for _ in range(args.warmup):
            cpu_oracle_prefill_rate(args.workload, n)
        qps, t, threads, sample = cpu_oracle_prefill_rate(args.workload, n,
                                                          steps=max(1, args.steps))
        line = {
            "impl": "reference", "metric": PREFILL_METRIC, "value": qps, "unit": "queries/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "n_q": spec["n_q"], "ctx": spec["ctx"],
                       "ratio": spec["ratio"], "key_fmt": spec["key_fmt"]},
            "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    n = args.cpu_sample or auto_cpu_sample(args.workload)
    for _ in range(args.warmup):
        cpu_oracle_rate(args.workload, n)
    qps, t, threads, sample = cpu_oracle_rate(args.workload, n, steps=max(1, args.steps))
    line = {
        "impl": "reference", "metric": METRIC, "value": qps, "unit": "queries/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch": spec["B"], "tokens": spec["T"],
                   "ratio": spec["ratio"], "key_fmt": spec["key_fmt"]},
        "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    __graft_entry__.build()
    import synth
    import two_tier_sparse_gb300 as dsa

    spec = dict(synth.WORKLOADS[args.workload])
    if spec["kind"] == "prefill":
        return run_prefill(args, spec, dsa, synth, dev, rank, world)
    if spec["kind"] == "multi":
        return run_multi(args, spec, dsa, synth, dev, rank, world)
    B, T, ratio, fmt = spec["B"], spec["T"], spec["ratio"], spec["key_fmt"]
    page_rows = spec.get("page_rows", 0)
    if args.batch:
        B = args.batch
    # Every rank decodes its own batch: seeds differ per rank.
    t0 = time.time()
    kv_fmt = spec.get("kv_fmt", "bf16")
    inp = synth.decode_inputs([T] * B, ratio, fmt, shard_seed(spec["seed"], rank), kv_fmt=kv_fmt)
    gen_s = time.time() - t0
    cfg = dsa.config(ratio=ratio, kv_fmt=dsa.KV_FP8_E4M3 if kv_fmt == "fp8" else dsa.KV_BF16,
                     kv_scale=inp.kv_scale)
    cap = inp.cap
    L = int(inp.n_latents.max())

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    q, q_idx, w = d(inp.q), d(inp.q_idx), d(inp.w)
    latents, swa = d(inp.latents), d(inp.swa)
    n_lat, swa_len = d(inp.n_latents), d(inp.swa_len)
    keys = dsa.Keys(fmt, d(inp.keys.data), None if inp.keys.scales is None else
                    d(inp.keys.scales))
    del inp
    pages = None
    if page_rows:
        # Every cache in pages of page_rows tokens: sequence b's logical page p
        # is physical page table[b, p] of a pool, a seeded permutation of the
        # B x cap / page_rows pages plus a few spare ones.
        pps = cap // page_rows
        n_pages = B * pps + 4
        gen = torch.Generator().manual_seed(shard_seed(spec["seed"], rank))
        table = torch.randperm(n_pages, generator=gen)[:B * pps].to(torch.int32).view(B, pps)
        flat = table.view(-1).to(dev, torch.int64)

        def paged(t):
            if t.dtype == torch.uint16:  # bf16 bit patterns: copied as int16
                t = t.view(torch.int16)
            pool = torch.zeros((n_pages * page_rows,) + tuple(t.shape[2:]), dtype=t.dtype,
                               device=dev)
            pool.view(n_pages, page_rows, *t.shape[2:])[flat] = t.view(B * pps, page_rows,
                                                                       *t.shape[2:])
            return pool
        pages = dsa.Pages(table.to(dev), page_rows, n_pages)
        latents = paged(latents)
        keys = dsa.Keys(fmt, paged(keys.data), None if keys.scales is None else
                        paged(keys.scales), pages)
        torch.cuda.empty_cache()
    nbc = cap // 8
    # block keys: [B, nbc, ...], or (paged) a pool of page_rows / 8 rows a page
    lead = (pages.c.n_pages * page_rows // 8,) if pages is not None else (B, nbc)
    if fmt == "bf16":
        pooled = dsa.Keys(fmt, torch.empty(lead + (128,), dtype=torch.int16, device=dev),
                          pages=pages)
    else:
        if pages is None and fmt == "mxfp4":
            lead = (B, nbc + (nbc & 1))  # MXFP4 rows are read in pairs
        width = 64 if fmt == "mxfp4" else 128
        pooled = dsa.Keys(fmt, torch.empty(lead + (width,), dtype=torch.uint8, device=dev),
                          torch.empty(lead + (4,), dtype=torch.uint8, device=dev), pages)
    ws = dsa.workspace(cfg, B, cap, dev)
    out = torch.empty((B, 64, 512), dtype=torch.int16, device=dev)
    lse = torch.empty((B, 64), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    # The pooled-key cache is built once (cache build, outside the step).
    dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws)
    torch.cuda.synchronize()

    def step():
        dsa.decode_step(cfg, q, q_idx, w, keys, pooled, latents, n_lat, cap, swa, swa_len, out,
                        ws, lse=lse, update_pool=True)

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")

    # The step is captured once in a CUDA graph (the graph keeps the launches'
    # programmatic edges) and each timed step is one replay. If the capture is
    # refused, the steps are launched on the stream instead and the line says so.
    graph = {"kernels_per_replay": None}
    g = None
    try:
        g = torch.cuda.CUDAGraph()
        dsa.launch_counts(reset=True)
        with torch.cuda.graph(g):
            step()
        per_replay = dsa.launch_counts(reset=True)
        graph["kernels_per_replay"] = int(sum(per_replay.values()))
        for _ in range(3):
            flush()
            g.replay()
        torch.cuda.synchronize()
    except RuntimeError as e:
        g = None
        graph["error"] = str(e).splitlines()[0][:200] if str(e) else type(e).__name__
    run = g.replay if g is not None else step
    graph["timed_launch"] = "cuda graph replay" if g is not None else "stream launches"

    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    dsa.launch_counts(reset=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # nvidia-smi samples every 100 ms: keep the GPU under the same load for
        # 1.5 s before the timed steps so the samples describe the timed region.
        t_end = time.time() + 1.5
        while time.time() < t_end:
            for _ in range(20):
                flush()
                run()
            torch.cuda.synchronize()
        dsa.launch_counts(reset=True)
        # Timed steps: events around each step only (an event between two
        # kernels would cut their programmatic overlap).
        for i in range(K):
            flush()
            ev_s[i].record()
            run()
            ev_e[i].record()
        torch.cuda.synchronize()
    counts = dsa.launch_counts(reset=True)
    if g is not None:  # replays launch the captured kernels without a host call each
        counts = {k: v * K for k, v in per_replay.items()}
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(ev_s, ev_e)]
    total_ms = float(sum(step_ms))
    total_ms = reduce_max([total_ms], dev)[0]
    ms_per_step = total_ms / K
    value = job_rate(B, world, ms_per_step)

    # Second timed pass, same steps, with CUDA events around every launch of the
    # library on the launching stream: the per-kernel breakdown and the scan's
    # per-launch durations for the roofline.
    kinds = {"pool": 1, "scan": 2, "select": 2, "attn": 1}
    kev = {k: ([torch.cuda.Event(enable_timing=True) for _ in range(n * K)],
               [torch.cuda.Event(enable_timing=True) for _ in range(n * K)])
           for k, n in kinds.items()}
    for k, (a_, b_) in kev.items():
        dsa.profile_events(k, a_, b_)
    for i in range(K):
        flush()
        step()
    torch.cuda.synchronize()
    for k in kinds:
        dsa.profile_events(k, [], [])
    n_launch = dsa.launch_counts(reset=True)
    kern_ms = {k: [s.elapsed_time(e) for s, e in zip(*kev[k])][:n_launch[k]] for k in kinds}
    kernel_ms = {k: float(sum(v) / K) for k, v in kern_ms.items()}
    scan_ms = kern_ms["scan"]

    # The same steps launched on the stream, one host call a step, timed the
    # same way: reported beside the graph-replay figure.
    # (Every rank runs this pass, so the ranks' collectives stay matched.)
    for i in range(K):
        flush()
        ev_s[i].record()
        step()
        ev_e[i].record()
    torch.cuda.synchronize()
    st_ms = reduce_max([sum(s.elapsed_time(e) for s, e in zip(ev_s, ev_e)) / K], dev)[0]
    graph["stream_launched"] = {"value": job_rate(B, world, st_ms), "unit": "queries/s",
                                "ms_per_step": st_ms}
    dsa.launch_counts(reset=True)

    # Stage costs inside a replay: CUDA graphs of growing prefixes of the step,
    # made of the C ABI's separate calls (tail pool + dsa_index_blocks, then
    # + dsa_topk, then + the attention), each timed like the step. The
    # per-kernel breakdown above brackets every launch with events, which adds
    # a launch's latency to each kernel and cuts their programmatic overlap.
    stages = {}
    try:
        nb_s = -(-L // 8)
        has_block = nb_s > cfg.k_blocks
        bids_p = torch.empty((B, cfg.k_blocks), dtype=torch.int32, device=dev)
        tids_p = torch.empty((B, cfg.k_tokens), dtype=torch.int32, device=dev)
        out_p = torch.empty_like(out)
        lse_p = torch.empty_like(lse)

        def p_pool():
            dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws, tail_only=True)

        def p_block():
            dsa.index_blocks(cfg, q_idx, w, pooled, n_lat, cap, bids_p, ws)

        def p_token():
            dsa.topk(cfg, q_idx, w, keys, bids_p if has_block else None, n_lat, cap, tids_p, ws)

        def p_attn():
            if pages is not None:
                dsa.sparse_attn_decode_paged(cfg, q, latents, pages, n_lat, tids_p, swa, swa_len,
                                             out_p, ws, lse=lse_p)
            else:
                dsa.sparse_attn_decode(cfg, q, latents, n_lat, tids_p, swa, swa_len, out_p, ws,
                                       lse=lse_p)

        first = [p_pool, p_block] if has_block else [p_pool]
        prefixes = [first, first + [p_token], first + [p_token, p_attn]]
        times = []
        for fns in prefixes:
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp):
                for f in fns:
                    f()
            for _ in range(3):
                flush()
                gp.replay()
            for i in range(K):
                flush()
                ev_s[i].record()
                gp.replay()
                ev_e[i].record()
            torch.cuda.synchronize()
            times.append(sum(s.elapsed_time(e) for s, e in zip(ev_s, ev_e)) / K)
        stages = {"pool + block stage" if has_block else "pool": times[0],
                  "token stage": times[1] - times[0], "attention": times[2] - times[1],
                  "all three prefixes' last (the calls one by one)": times[2],
                  "how": "CUDA graphs of growing prefixes of the step made of the C ABI's "
                         "separate calls; a stage is the difference of two prefixes' replay "
                         "times (ms)"}
    except RuntimeError as e:
        stages = {"error": str(e).splitlines()[0][:200] if str(e) else type(e).__name__}
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")
    dsa.launch_counts(reset=True)

    # Roofline of the dominant kernel: the indexer scan. Algorithmic bytes per
    # launch = rows scanned x bytes per key row (MXFP8: 128 codes + 4 scale
    # bytes; MXFP4: 64 + 4; bf16: 256); both launches of a step scan 2048 x 8 = 16384 rows per
    # query (16384 block keys, then 16384 candidate latents).
    row_bytes = {"mxfp8": 132, "mxfp4": 68}.get(fmt, 256)
    nb = -(-L // 8)
    blk_rows = nb if nb > cfg.k_blocks else 0
    tok_rows = 8 * cfg.k_blocks if nb > cfg.k_blocks else L
    per_launch = [B * blk_rows * row_bytes, B * tok_rows * row_bytes] if blk_rows else \
        [B * tok_rows * row_bytes]
    launches_per_step = len(per_launch)
    bytes_per_launch = float(np.mean(per_launch))
    scan_avg_ms = float(np.mean(scan_ms)) if scan_ms else float("nan")
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = bytes_per_launch / (scan_avg_ms * 1e-3) / 1e9
    # whole-step algorithmic bytes (keys scanned + latent rows gathered + window + q/out;
    # a latent or window row is 1024 bytes in bf16, 512 in fp8)
    kv_row = 512 if kv_fmt == "fp8" else 1024
    step_bytes = B * (blk_rows * row_bytes + tok_rows * row_bytes + 512 * kv_row + 128 * kv_row
                      + 64 * 512 * 2 * 2 + 16 * 128 * 2)
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "scan_traffic.json")
    if os.path.exists(tr_path):
        try:
            tr = json.load(open(tr_path))
            if tr.get("workload") == args.workload:
                traffic = tr.get("dram_bytes_per_launch")
        except Exception:
            traffic = None

    # End to end through the C ABI with host buffers: each step's inputs (q,
    # q_idx, w) travel in one copy from a pinned staging buffer and its
    # results (out, lse) come back in one copy, as a serving loop would stage
    # them.
    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, n

    def views(buf, tensors, offs):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for t, o in zip(tensors, offs)]

    in_offs, in_n = packed([q, q_idx, w])
    in_h = torch.empty(in_n, dtype=torch.uint8).pin_memory()
    for v, t in zip(views(in_h, [q, q_idx, w], in_offs), [q, q_idx, w]):
        v.copy_(t.cpu())
    in_d = torch.empty(in_n, dtype=torch.uint8, device=dev)
    q_d, qi_d, w_d = views(in_d, [q, q_idx, w], in_offs)
    out_offs, out_n = packed([out, lse])
    res_d = torch.empty(out_n, dtype=torch.uint8, device=dev)
    out_d, lse_d = views(res_d, [out, lse], out_offs)
    res_h = torch.empty(out_n, dtype=torch.uint8).pin_memory()

    def e2e_step():
        in_d.copy_(in_h, non_blocking=True)
        dsa.decode_step(cfg, q_d, qi_d, w_d, keys, pooled, latents, n_lat, cap, swa, swa_len,
                        out_d, ws, lse=lse_d, update_pool=True)
        res_h.copy_(res_d, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush()
        e_s[i].record()
        e2e_step()
        e_e[i].record()
    torch.cuda.synchronize()
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / K

    # Pipelined, as a serving loop runs: step i + 1's inputs go in (one copy
    # stream) while step i computes, and step i's results come back (a second
    # copy stream) while step i + 1 computes; staging is double-buffered on
    # the device. One timed region over K steps with no L2 flush inside it:
    # each step reads ~330 MB out of 9.6 GB of caches, far more than the
    # 129 MB L2, so nothing useful carries over from one step to the next.
    main = torch.cuda.current_stream(dev)
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_bufs = [in_d, torch.empty_like(in_d)]
    in_vs = [views(b_, [q, q_idx, w], in_offs) for b_ in in_bufs]
    res_bufs = [res_d, torch.empty_like(res_d)]
    res_vs = [views(b_, [out, lse], out_offs) for b_ in res_bufs]
    res_hs = [res_h, torch.empty(out_n, dtype=torch.uint8).pin_memory()]

    def run_pipelined(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_back = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        cs_in.wait_stream(main)
        cs_out.wait_stream(main)
        for i in range(n):
            k = i & 1
            with torch.cuda.stream(cs_in):
                if i >= 2:
                    cs_in.wait_event(ev_done[i - 2])  # step i - 2 has read in_bufs[k]
                in_bufs[k].copy_(in_h, non_blocking=True)
                ev_in[i].record(cs_in)
            main.wait_event(ev_in[i])
            if i >= 2:
                main.wait_event(ev_back[i - 2])  # res_bufs[k] has been copied out
            qv, qiv, wv = in_vs[k]
            ov, lv = res_vs[k]
            dsa.decode_step(cfg, qv, qiv, wv, keys, pooled, latents, n_lat, cap, swa, swa_len, ov,
                            ws, lse=lv, update_pool=True)
            ev_done[i].record(main)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(ev_done[i])
                res_hs[k].copy_(res_bufs[k], non_blocking=True)
                ev_back[i].record(cs_out)
        main.wait_stream(cs_out)
        t1.record(main)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    run_pipelined(3)
    e2e_pipe_ms = run_pipelined(K)
    e2e_ms, e2e_pipe_ms = reduce_max([e2e_ms, e2e_pipe_ms], dev)
    h2d = in_n   # bytes of the one input copy (q, q_idx, w, each padded to 256 B)
    d2h = out_n  # bytes of the one result copy (out, lse)
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        n = args.cpu_sample or auto_cpu_sample(args.workload)
        qps, t, threads, sample = cpu_oracle_rate(args.workload, n)
        cpu = {"value": qps, "unit": "queries/s", "cores": threads, "kind": "oracle",
               "sample": sample, "threads_note": THREADS_NOTE,
               "one_thread": cpu_oracle_one_thread(args.workload, max(1, min(n, 4)))}
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch_per_gpu": B, "tokens": T, "ratio": ratio,
                   "latents": L, "blocks": nb, "k_blocks": cfg.k_blocks,
                   "layout": f"paged, {page_rows}-token pages" if page_rows else "contiguous",
                   "k_tokens": cfg.k_tokens, "window": cfg.window, "key_fmt": fmt,
                   "kv_fmt": kv_fmt,
                   "l2": L2Flush.DESCRIPTION,
                   "step_algorithmic_bytes": step_bytes,
                   "step_hbm_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
                   "step_hbm_frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak,
                   "input_gen_s": round(gen_s, 1)},
        "roofline": {"kernel": "scan (indexer scores, tcgen05)", "bound": "hbm",
                     "launch_ms_block_stage": float(np.mean(scan_ms[0::2])) if blk_rows else None,
                     "launch_ms_token_stage": float(np.mean(scan_ms[1::2] if blk_rows else scan_ms)),
                     "achieved": achieved, "peak": hbm_peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "avg_launch_ms": scan_avg_ms, "launches_per_step": launches_per_step},
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(B, world, e2e_pipe_ms), "unit": "queries/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_pipe_ms,
                "mode": "pipelined: each step's input copy and result copy overlap the "
                        "neighbouring steps' compute; one timed region over the steps, "
                        "no L2 flush inside it",
                "serial": {"value": job_rate(B, world, e2e_ms), "ms_per_step": e2e_ms,
                           "mode": "copy in, step, copy out; L2 flushed before each step"}},
        "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
        "graph": graph,
        "kernel_ms_per_step": kernel_ms,
        "stage_ms_in_graph": stages,
        "gpu_launches": int(sum(counts.values())),
        "gpu_launches_by_kind": counts,
        "clocks": clocks.summary(),
    }
    if args.workload == DEFAULT_WORKLOAD and not args.no_prefill and world == 1 and not args.batch:
        # The prefill chunk's line rides along under extra.prefill, measured in
        # the same run (its own timing rules, clocks and CPU figure).
        pspec = dict(synth.WORKLOADS[PREFILL_WORKLOAD])
        pspec.pop("kind")
        line["extra"] = {"prefill": run_prefill(args, pspec, dsa, synth, dev, rank, world,
                                                workload=PREFILL_WORKLOAD,
                                                steps=min(K, 10), emit=False)}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# Algorithmic flops per prefill query (multiply-adds x 2): the block scan over
# the visible blocks, the token scan over the kept tokens, QK^T and PV.
def prefill_flops(n_q: int, ctx: int, ratio: int, k_blocks: int = 2048, k_tokens: int = 512,
                  window: int = 128) -> float:
    total = 0.0
    for i in range(n_q):
        p = ctx + i
        n_vis = (p + 1) // ratio
        nb = (n_vis + 7) // 8
        kept = min(nb, k_blocks)
        tokens = min(n_vis, kept * 8)
        rows = min(tokens, k_tokens) + min(window, p + 1)
        total += 2.0 * 16 * 128 * (nb + tokens) + 2.0 * 2 * 64 * 512 * rows
    return total


def prefill_executed_flops(n_q: int, ctx: int, ratio: int, k_blocks: int = 2048,
                           k_tokens: int = 512, window: int = 128) -> float:
    """Flops the tensor cores execute for a prefill chunk, padding included.

    The batched scans run one M=128 x N=256 x K=128 MMA per 128-row tile for
    each group of 16 queries. The block stage covers every complete block of
    the chunk's context; the token stage covers the visible latents of the
    group's last query, rounded up to whole blocks. Attention runs 64-row
    tiles: QK^T at M=128 (64 heads in half the rows, N=64 rows, K=512) and PV
    as four M=128 latent slices (N=64 heads, K=64 rows).
    """
    n_lat = (ctx + n_q) // ratio
    lat_cols = -(-n_lat // 8) * 8
    blk_tiles = -(-(n_lat // 8) // 128)
    per_tile = 2.0 * 128 * 256 * 128
    total = 0.0
    for g0 in range(0, n_q, 16):
        vis = (ctx + min(g0 + 16, n_q)) // ratio  # the group's last query, at ctx + min(...) - 1
        cover = min(-(-vis // 8) * 8, lat_cols)
        total += (blk_tiles + -(-cover // 128)) * per_tile
    for i in range(n_q):
        p = ctx + i
        n_vis = (p + 1) // ratio
        tokens = min(n_vis, min((n_vis + 7) // 8, k_blocks) * 8)
        rows = min(tokens, k_tokens) + min(window, p + 1)
        total += (-(-rows // 64) * 64) * (2.0 * 128 * 512 + 2.0 * 512 * 64)
    return total


def run_prefill(args, spec, dsa, synth, dev, rank, world, workload=None, steps=None,
                emit=True):
    """A prefill chunk per step: n_q causal queries appended to ctx tokens of
    one sequence (cache build, i.e. the pooled keys, outside the step).
    Returns rank 0's JSON line (printed when `emit`)."""
    import torch
    workload = workload or args.workload
    n_q, ctx, ratio, fmt = spec["n_q"], spec["ctx"], spec["ratio"], spec["key_fmt"]
    if args.batch and emit:
        n_q = args.batch  # a smaller chunk (profiling); the line then names it in config
    t0 = time.time()
    pf = synth.prefill_inputs(n_q, ctx, ratio, fmt, shard_seed(spec["seed"], rank))
    gen_s = time.time() - t0
    cfg = dsa.config(ratio=ratio)
    n_lat = (ctx + n_q) // ratio

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    q, q_idx, w, latents, swa = d(pf.q), d(pf.q_idx), d(pf.w), d(pf.latents), d(pf.swa)
    keys = dsa.Keys(fmt, d(pf.keys.data), None if pf.keys.scales is None else d(pf.keys.scales))
    del pf
    nbf = n_lat // 8
    if fmt == "bf16":
        pooled = dsa.Keys(fmt, torch.zeros((1, max(nbf, 1), 128), dtype=torch.int16, device=dev))
    else:
        pooled = dsa.Keys(fmt, torch.zeros((1, max(nbf, 1), 128), dtype=torch.uint8, device=dev),
                          torch.zeros((1, max(nbf, 1), 4), dtype=torch.uint8, device=dev))
    ws = dsa.workspace(cfg, n_q, n_lat, dev)
    keys1 = dsa.Keys(fmt, keys.data[None], None if keys.scales is None else keys.scales[None])
    dsa.pool_index_keys(cfg, keys1, torch.tensor([nbf * 8], dtype=torch.int32, device=dev),
                        nbf * 8, pooled, ws)
    pooled2 = dsa.Keys(fmt, pooled.data[0], None if pooled.scales is None else pooled.scales[0])
    out = torch.empty((n_q, 64, 512), dtype=torch.int16, device=dev)
    lse = torch.empty((n_q, 64), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)

    def step():
        dsa.sparse_attn_prefill(cfg, ctx, q, q_idx, w, latents, keys, pooled2, swa, out, ws, lse=lse)

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")
    K = steps or args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    dsa.launch_counts(reset=True)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clocks:
        t_end = time.time() + 1.5
        while time.time() < t_end:
            flush()
            step()
            torch.cuda.synchronize()
        dsa.launch_counts(reset=True)
        for i in range(K):
            flush()
            ev_s[i].record()
            step()
            ev_e[i].record()
        torch.cuda.synchronize()
    counts = dsa.launch_counts(reset=True)
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(ev_s, ev_e)]
    ms = reduce_max([float(np.mean(step_ms))], dev)[0]
    # per-kernel breakdown (second pass with events around each launch)
    kinds = {"pool": 1, "scan": 2, "select": 2, "attn": 1, "other": 1}
    kev = {k: ([torch.cuda.Event(enable_timing=True) for _ in range(n * K)],
               [torch.cuda.Event(enable_timing=True) for _ in range(n * K)])
           for k, n in kinds.items()}
    for k, (a_, b_) in kev.items():
        dsa.profile_events(k, a_, b_)
    for i in range(K):
        flush()
        step()
    torch.cuda.synchronize()
    for k in kinds:
        dsa.profile_events(k, [], [])
    n_launch = dsa.launch_counts(reset=True)
    kernel_ms = {k: float(sum(s_.elapsed_time(e_) for s_, e_ in list(zip(*kev[k]))[:n_launch[k]]) / K)
                 for k in kinds}
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")
    flops = prefill_flops(n_q, ctx, ratio)
    exec_flops = prefill_executed_flops(n_q, ctx, ratio)
    _, tf_peak, peak_kind = measured_peaks()
    tf_sus = sustained_bf16_peak()
    tflops = flops / (ms * 1e-3) / 1e12
    exec_tflops = exec_flops / (ms * 1e-3) / 1e12
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            qps, _, threads, sample = cpu_oracle_prefill_rate(
                workload, (args.cpu_sample if emit else 0) or PREFILL_CPU_SAMPLE)
            cpu = {"value": qps, "unit": "queries/s", "cores": threads, "kind": "oracle",
                   "sample": sample, "threads_note": THREADS_NOTE}
        line = {
            "metric": PREFILL_METRIC,
            "value": job_rate(n_q, world, ms), "unit": "queries/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload, "n_q": n_q, "ctx": ctx, "ratio": ratio,
                       "key_fmt": fmt, "latents": n_lat,
                       "l2": L2Flush.DESCRIPTION,
                       "input_gen_s": round(gen_s, 1)},
            "roofline": {"kernel": "whole prefill step (tensor-core contractions)", "bound": "tensor",
                         "achieved": tflops, "peak": tf_peak, "peak_kind": peak_kind,
                         "unit": "TFLOP/s", "frac": tflops / tf_peak,
                         "algorithmic_flops_per_step": flops,
                         "frac_of_sustained": tflops / tf_sus if tf_sus else None,
                         "sustained_peak": tf_sus,
                         "executed_flops_per_step": exec_flops,
                         "executed_tflops": exec_tflops,
                         "executed_frac": exec_tflops / tf_peak},
            "cpu_baseline": cpu,
            "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q_)) for q_ in (10, 50, 90)],
            "kernel_ms_per_step": kernel_ms,
            "gpu_launches": int(sum(counts.values())),
            "gpu_launches_by_kind": counts,
            "clocks": clocks.summary(),
        }
        if emit:
            print(json.dumps(line), flush=True)
    if world > 1 and emit:
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


def run_multi(args, spec, dsa, synth, dev, rank, world):
    """Multi-query decode: every sequence's n_q queries at its last n_q
    positions, one dsa_decode_multi call a step (inputs resident in HBM, the
    block-key cache built once outside the step)."""
    import torch
    B, T, n_q, ratio, fmt = spec["B"], spec["T"], spec["n_q"], spec["ratio"], spec["key_fmt"]
    if args.batch:
        B = args.batch
    t0 = time.time()
    m = synth.multi_inputs([T] * B, n_q, ratio, fmt, shard_seed(spec["seed"], rank))
    gen_s = time.time() - t0
    cfg = dsa.config(ratio=ratio)
    cap = m.cap

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    q, q_idx, w, latents, swa = d(m.q), d(m.q_idx), d(m.w), d(m.latents), d(m.swa)
    n_tok, n_lat = d(m.T.astype(np.int32)), d(m.n_latents)
    keys = dsa.Keys(fmt, d(m.keys.data), None if m.keys.scales is None else d(m.keys.scales))
    L = int(m.n_latents.max())
    del m
    nbc = cap // 8
    width = 64 if fmt == "mxfp4" else 128
    nbc += nbc & 1 if fmt == "mxfp4" else 0
    if fmt == "bf16":
        pooled = dsa.Keys(fmt, torch.empty((B, nbc, 128), dtype=torch.int16, device=dev))
    else:
        pooled = dsa.Keys(fmt, torch.empty((B, nbc, width), dtype=torch.uint8, device=dev),
                          torch.empty((B, nbc, 4), dtype=torch.uint8, device=dev))
    ws = dsa.workspace(cfg, B * n_q, cap, dev)
    dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws)
    out = torch.empty((B, n_q, 64, 512), dtype=torch.int16, device=dev)
    lse = torch.empty((B, n_q, 64), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)

    def step():
        dsa.decode_multi(cfg, n_tok, q, q_idx, w, keys, pooled, latents, cap, swa, out, ws, lse=lse)

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")
    g = torch.cuda.CUDAGraph()
    dsa.launch_counts(reset=True)
    with torch.cuda.graph(g):
        step()
    per_replay = dsa.launch_counts(reset=True)
    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clocks:
        t_end = time.time() + 1.5
        while time.time() < t_end:
            for _ in range(10):
                flush()
                g.replay()
            torch.cuda.synchronize()
        for i in range(K):
            flush()
            ev_s[i].record()
            g.replay()
            ev_e[i].record()
        torch.cuda.synchronize()
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(ev_s, ev_e)]
    ms = reduce_max([float(np.mean(step_ms))], dev)[0]
    kinds = {"pool": 1, "scan": 2, "select": 2, "attn": 1}
    kev = {k: ([torch.cuda.Event(enable_timing=True) for _ in range(n * K)],
               [torch.cuda.Event(enable_timing=True) for _ in range(n * K)])
           for k, n in kinds.items()}
    for k, (a_, b_) in kev.items():
        dsa.profile_events(k, a_, b_)
    dsa.launch_counts(reset=True)
    for i in range(K):
        flush()
        step()
    torch.cuda.synchronize()
    for k in kinds:
        dsa.profile_events(k, [], [])
    n_launch = dsa.launch_counts(reset=True)
    kern_ms = {k: [s_.elapsed_time(e_) for s_, e_ in zip(*kev[k])][:n_launch[k]] for k in kinds}
    kernel_ms = {k: float(sum(v) / K) for k, v in kern_ms.items()}
    code, info = dsa.read_device_status(ws)
    if code != 0:
        raise SystemExit(f"device status {code} info {info:#x}")
    # Scan roofline. Every query scans its sequence's block keys and its own
    # 2048 candidate blocks; the n_q queries of a sequence read the same block
    # keys, so the algorithmic bytes count those once per sequence (the
    # candidate blocks, mostly shared too, are counted per query: an upper
    # bound of the unique bytes).
    row_bytes = {"mxfp8": 132, "mxfp4": 68}.get(fmt, 256)
    nb = -(-L // 8)
    blk_bytes = B * nb * row_bytes
    tok_bytes = B * n_q * min(nb, cfg.k_blocks) * 8 * row_bytes
    scan_ms = kern_ms["scan"]
    hbm_peak, _, peak_kind = measured_peaks()
    achieved_blk = blk_bytes / (float(np.mean(scan_ms[0::2])) * 1e-3) / 1e9
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            qps, _, threads, sample = cpu_oracle_multi_rate(args.workload, args.cpu_sample or 2)
            cpu = {"value": qps, "unit": "queries/s", "cores": threads, "kind": "oracle",
                   "sample": sample, "threads_note": THREADS_NOTE}
        line = {
            "metric": MULTI_METRIC, "value": job_rate(B * n_q, world, ms), "unit": "queries/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": args.workload, "batch_per_gpu": B, "queries_per_seq": n_q,
                       "tokens": T, "ratio": ratio, "key_fmt": fmt, "latents": L,
                       "l2": L2Flush.DESCRIPTION, "input_gen_s": round(gen_s, 1)},
            "roofline": {"kernel": "scan, block stage (the block keys shared by a sequence's "
                                   "queries, counted once)", "bound": "hbm",
                         "achieved": achieved_blk, "peak": hbm_peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": achieved_blk / hbm_peak, "traffic": None,
                         "algorithmic_bytes_per_launch": blk_bytes,
                         "token_stage_bytes_upper_bound": tok_bytes,
                         "launch_ms_block_stage": float(np.mean(scan_ms[0::2])),
                         "launch_ms_token_stage": float(np.mean(scan_ms[1::2]))},
            "cpu_baseline": cpu,
            "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q_)) for q_ in (10, 50, 90)],
            "kernel_ms_per_step": kernel_ms,
            "gpu_launches": int(sum(per_replay.values())) * K,
            "gpu_launches_by_kind": {k: v * K for k, v in per_replay.items()},
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
