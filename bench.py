#!/usr/bin/env python
"""Benchmark: paged decode attention KV GB/s (% of GB300 HBM peak) and decode steps/s.

A *step* is one decode step of the 16-layer engine's attention hot path: for
every layer, the RoPE + page-slot append of each sequence's new token, then
paged GQA decode attention over the sequence's pages with the log-sum-exp merge
of its chunks -- by default one fused kernel per layer (``--path separate``: the
two named calls, pkv_append_rope then pkv_decode_attention; ``--split-merge``:
the attention's two-kernel form).  Default workload ``b256``: batch 256, every sequence at 2,048 tokens
(128 pages per sequence and layer), 32 query / 8 KV heads, head_dim 64, BF16 KV
pool of 524,288 pages (16 GiB).  Other workloads: ``--config b64`` (log-normal
lengths, median 300) and ``--config b8`` (uniform lengths).

The timed region replays CUDA graphs of whole steps; the inputs (17 GB of KV per
b256 step) are far larger than the 129 MB L2, so no flush is needed.  A second
pass replays the same steps from graphs in which every attention launch is
bracketed by external timing events; these give the dominant kernel's average
duration for the roofline (the step time itself comes from uninstrumented
graphs, since an event between two launches would serialise their programmatic
dependent launch).

The default run also measures further configurations (``--extra``: the ragged
batch 64, batch 8, the separate calls on batch 64, FP8 pages on batch 64 and
256) and reports them under ``configs``; a read-only HBM probe gives the
streaming ceiling the fractions are also reported against.  The CPU baseline is
the FP64 oracle on the GPU batch's own inputs, single-threaded and on every
host core.

``--impl reference`` times the FP64 CPU oracle on a bounded sample of the same
workload on the host cores (the reference arm; it runs none of the CUDA path).

Multi-GPU (``torchrun --nproc-per-node N``): independent replicas, one per GPU,
each with its own batch (weak scaling); the max elapsed time over ranks is used.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and decode steps/s"
CONFIG_TEXT = {
    "b256": "long-context batch 256: every sequence 2048 tokens (128 pages), 16 layers, 32 Q / 8 KV heads, "
            "head_dim 64, pool of 524288 pages (32 KiB BF16 or 17 KiB FP8 each), random page permutation",
    "b64": "ragged batch 64: log-normal lengths (median 300, sigma 1, clipped to [1, 2048], boundary lengths "
           "1/16/17/32/33/2048 included), 16 layers, 1% of keys x8, 4096 pages per layer",
    "b8": "batch 8: lengths uniform in [1, 2048], 16 layers, 4096 pages of 32 KiB per layer",
    "trace": "continuous-batching trace: 500 steps, Poisson(0.6) arrivals per step, prompts U[8,1024], output "
             "budgets U[16,1024], contexts <= 2048, batch cap 192, 16 layers, page-budget admission, prefill "
             "page fill, lazy pages",
}
VARIANTS = {"default": 0, "simt": 1, "mma": 2}
# Per-workload launch settings (pages per unit, ring depth, sorted dispatch, micro-batch
# chains), chosen by measurement; the full-size parity tests run the same ones.
from paged_kv_decode_12_gb300 import launch as LAUNCH  # noqa: E402  (no torch import)

DEFAULT_CHUNK = {k: v for k, v in LAUNCH.CHUNK.items() if k != "tiny"}
DEFAULT_RING = {k: v for k, v in LAUNCH.RING.items() if k != "tiny"}
DEFAULT_SORTED = {k: v for k, v in LAUNCH.SORTED.items() if k != "tiny"}
DEFAULT_RING_FP8 = {k: v for k, v in LAUNCH.RING_FP8.items() if k != "tiny"}
DEFAULT_CHAINS = {k: v for k, v in LAUNCH.CHAINS.items() if k != "tiny"}
DEFAULT_CHAINS_FP8 = {k: v for k, v in LAUNCH.CHAINS_FP8.items() if k != "tiny"}
L2_BYTES = 129 * 10**6


# --------------------------------------------------------------------------- distributed helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(base_seed: int, rank: int) -> int:
    """Each replica draws its own batch (weak scaling): seed offset by rank."""
    return base_seed + 1000 * rank


# --------------------------------------------------------------------------- peaks, clocks, profiles

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.6)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, power, reasons = [], None, [], set()
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# the sources the fused step kernels are built from (kernels, policies, tensor maps)
KERNEL_SOURCES = ("pkv_device.cuh", "pkv_fp8.cuh", "pkv_step.cu", "pkv_host.cpp", "pkv_internal.h")


def kernel_source_digest() -> str:
    """Digest of the attention kernels' sources (ties a stored ncu figure to the code it measured)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_decode_12_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(config: str, path: str, variant_name: str, pages_per_chunk: int, ring: int,
                     kv: str = "bf16", chains: int = 1, sorted_units: bool = False, split_merge: bool = False):
    """DRAM bytes per attention launch from the committed ncu summary
    (profiles/decode_traffic.json), if it was taken on the current kernel source;
    else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
            entries = json.load(f)
    except Exception:
        return None
    digest = kernel_source_digest()
    for e in entries:
        if (e.get("config") == config and e.get("path") == path and e.get("variant") == variant_name and
                e.get("pages_per_chunk") == pages_per_chunk and e.get("ring", 4) == ring and
                e.get("kv", "bf16") == kv and e.get("chains", 1) == chains and
                e.get("sorted_units", False) == sorted_units and e.get("split_merge", False) == split_merge and
                e.get("kernel_source_sha") == digest):
            return e.get("dram_bytes_per_launch")
    return None


# --------------------------------------------------------------------------- CPU oracle baseline

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_samples(w, n_seqs: int, seed: int, kv: str = "bf16"):
    """Host-side synthetic inputs for ``n_seqs`` sequences of one layer of workload ``w``
    (same length mix), each in its own small paged pool (FP8 pools: codes drawn as for the
    GPU workloads, N(0, 128^2) converted to E4M3, row scales uniform in [0.005, 0.009]).
    The reference arm uses these: it runs on the host cores only."""
    import oracle
    from paged_kv_decode_12_gb300 import workloads as wl

    rng = np.random.default_rng(seed)
    idx = rng.choice(w.batch, size=min(n_seqs, w.batch), replace=False)
    out = []
    for b in idx:
        L = int(w.seq_lens[b])
        npg = -(-L // wl.PAGE_SIZE)
        if kv == "fp8":
            pool = np.empty(npg * oracle.FP8_PAGE_BYTES, dtype=np.uint8)
            units = pool.reshape(npg, wl.NUM_KV_HEADS, -1)
            ncode = 2 * wl.PAGE_SIZE * wl.HEAD_DIM
            units[:, :, :ncode] = oracle.e4m3_from_f64(
                np.clip(rng.standard_normal((npg, wl.NUM_KV_HEADS, ncode)) * 128.0, -448, 448))
            units[:, :, ncode:].view(np.float32)[:] = rng.uniform(0.005, 0.009, (npg, wl.NUM_KV_HEADS,
                                                                                 2 * wl.PAGE_SIZE))
        else:
            pool = wl.bf16_normal_host(rng, (npg * 2 * wl.NUM_KV_HEADS * wl.PAGE_SIZE * wl.HEAD_DIM,))
        bt = wl.permutation_block_tables(rng, [L], npg, w.max_blocks)
        out.append(dict(L=L, npg=npg, pool=pool, bt=bt,
                        q=wl.bf16_normal_host(rng, (1, wl.NUM_Q_HEADS, wl.HEAD_DIM)),
                        k_new=wl.bf16_normal_host(rng, (1, wl.NUM_KV_HEADS, wl.HEAD_DIM)),
                        v_new=wl.bf16_normal_host(rng, (1, wl.NUM_KV_HEADS, wl.HEAD_DIM))))
    return out


# (layers, sequences) of the GPU batch the CPU baseline runs, per workload: whole steps
# where the oracle finishes them in seconds, else a stated fraction of one step
CPU_SAMPLE = {"tiny": (None, None), "b8": (None, None), "b64": (1, None), "b256": (1, 32)}


def gpu_batch_sample(dw, kv: str):
    """Oracle inputs copied from the GPU batch itself (so the CPU baseline runs the very
    inputs the GPU step runs): per (layer, sequence) of ``CPU_SAMPLE``, the sequence's
    pages from the device pool, its block-table row renumbered into that small pool, and
    its unrotated q, k_new, v_new rows.  Returns (samples, fraction of one step)."""
    import torch

    from paged_kv_decode_12_gb300 import workloads as wl

    w = dw.w
    n_layers, n_seqs = CPU_SAMPLE.get(w.name, (1, 8))
    layers = range(w.layers if n_layers is None else min(n_layers, w.layers))
    seqs = range(w.batch if n_seqs is None else min(n_seqs, w.batch))
    page_bytes = dw.eng.page_bytes
    pages_view = dw.eng.slab.view(dw.eng.num_pages, page_bytes)
    q0, k_new, v_new = (t.view(torch.int16).cpu().numpy().view(np.uint16) for t in (dw.q0, dw.k_new, dw.v_new))
    out = []
    for l in layers:
        for b in seqs:
            L = int(w.seq_lens[b])
            npg = -(-L // wl.PAGE_SIZE)
            ids = torch.from_numpy(dw.eng.bt_host[l, b, :npg].astype(np.int64)).to(pages_view.device)
            mini = pages_view[ids].cpu().numpy().reshape(-1)
            pool = mini.copy() if kv == "fp8" else mini.view(np.uint16).copy()
            bt = np.full((1, w.max_blocks), -1, dtype=np.int32)
            bt[0, :npg] = np.arange(npg)
            out.append(dict(L=L, npg=npg, pool=pool, bt=bt, q=q0[l, b][None].copy(), k_new=k_new[l, b][None].copy(),
                            v_new=v_new[l, b][None].copy()))
    frac = len(out) / (w.layers * w.batch)
    return out, frac


def oracle_run_one(s, kv: str = "bf16") -> int:
    """One oracle pass (append + attention, all 32 heads) over one sampled sequence;
    returns the KV tokens attended."""
    import oracle
    from paged_kv_decode_12_gb300 import workloads as wl

    append, decode = (oracle.append_fp8, oracle.decode_fp8) if kv == "fp8" else (oracle.append, oracle.decode)
    g = oracle.geom(s["npg"])
    q = s["q"].copy()
    append(s["pool"], g, s["bt"], [s["L"] - 1], s["k_new"], s["v_new"], q)
    decode(s["pool"], g, s["bt"], [s["L"]], q, 1.0 / math.sqrt(wl.HEAD_DIM))
    return s["L"]


def oracle_run_sample(sample, kv: str = "bf16", threads: int = 1) -> int:
    """Every sampled sequence once, on ``threads`` host threads (the C oracle releases the
    interpreter lock, and each sequence has its own pages); returns the KV tokens attended."""
    if threads <= 1:
        return sum(oracle_run_one(s, kv) for s in sample)
    import concurrent.futures

    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        return sum(ex.map(lambda s: oracle_run_one(s, kv), sample))


def time_oracle(sample, kv: str, threads: int, min_seconds: float):
    """Whole passes over the sample until ``min_seconds`` have elapsed: (KV GB/s, passes, s)."""
    from paged_kv_decode_12_gb300 import workloads as wl

    per_token = wl.kv_bytes_per_token(1, kv=kv)
    tokens, passes = 0, 0
    t0 = time.perf_counter()
    while True:
        tokens += oracle_run_sample(sample, kv, threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            return tokens * per_token / dt / 1e9, passes, dt


def cpu_baseline(dw, seconds: float, kv: str = "bf16") -> dict:
    """The FP64 oracle on the host cores, on the GPU batch's own inputs: single-threaded and
    with one thread per host core; ``value`` is the all-cores figure."""
    sample, frac = gpu_batch_sample(dw, kv)
    cores = host_cores()
    one, n1, t1 = time_oracle(sample, kv, 1, seconds * 0.5)
    many, nn, tn = time_oracle(sample, kv, cores, seconds * 0.5)
    w = dw.w
    what = (f"{len(sample)} (layer, sequence) pairs of the GPU batch ({frac:.4g} of one {w.layers}-layer step of "
            f"{w.name}; {sum(s['L'] for s in sample)} KV tokens): append + attention for all 32 query heads, "
            f"FP64 C oracle on the inputs the GPU step runs")
    return {"value": many, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{what}; {nn} passes on {cores} threads in {tn:.1f} s",
            "fraction_of_step": frac, "host_cores": cores,
            "single_thread": {"value": one, "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} passes on one thread in {t1:.1f} s"}}


# --------------------------------------------------------------------------- read-only HBM ceiling

def read_ceiling(device, gib: int = 4, reps: int = 5) -> dict:
    """Best read-only streaming rate of the device's HBM: libpkv's two read probes (16-byte
    loads; TMA bulk copies into shared memory) over a buffer far larger than L2, each at a
    few CTA counts, CUDA events on the launching stream, best of ``reps``."""
    import torch

    from paged_kv_decode_12_gb300 import pkv

    nbytes = gib << 30
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    buf.random_(0, 256)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    sink = torch.zeros(sms * 4 + 1, dtype=torch.int32, device=device)
    results = {}
    for name, fn, ctas in (("ldg", pkv.pkv_probe_read_ldg, (1, 2, 4)), ("bulk", pkv.pkv_probe_read_bulk, (1, 2))):
        for c in ctas:
            fn(buf, nbytes, sink, c)   # warm
            best = 0.0
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn(buf, nbytes, sink, c)
                b.record()
                torch.cuda.synchronize()
                best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
            results[f"{name}_{c}"] = best
    if int(sink[-1].item()) != 0:
        raise SystemExit("read probe: a bounded wait gave up")
    del buf
    torch.cuda.empty_cache()
    top = max(results, key=results.get)
    return {"gbs": results[top], "best_probe": top, "probes": results,
            "how": f"libpkv read probes over {gib} GiB (16-byte loads; TMA bulk copies of 32 KiB), best of {reps} "
                   "per probe and CTA count, CUDA events"}


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal


def config_block(w, a, variant_name: str, graph: bool) -> dict:
    """The ``config`` object of a JSON line; ``a`` holds one run's launch settings."""
    kv = w.kv_bytes_per_step(getattr(a, "kv", "bf16"))
    return {"workload": f"{a.config}: {CONFIG_TEXT[a.config]}", "batch": w.batch, "layers": w.layers,
            "seq_len_max": int(w.seq_lens.max()), "seq_len_mean": float(w.seq_lens.mean()),
            "pages_per_chunk": a.pages_per_chunk, "kernel_variant": variant_name, "cuda_graph": graph,
            "path": getattr(a, "path", "fused"), "pdl": not getattr(a, "no_pdl", False),
            "ring": getattr(a, "ring", 0), "sorted_units": getattr(a, "sorted", False),
            "split_merge": getattr(a, "split_merge", False),
            "chains": getattr(a, "chains", 1),
            "pipelined": getattr(a, "pipelined", False),
            "steps_per_graph": getattr(a, "steps_per_graph", None) if graph else None,
            "kv_pages": getattr(a, "kv", "bf16"),
            "kv_bytes_per_step": kv,
            "l2": f"inputs larger than L2 ({kv / 1e9:.2f} GB of KV per step vs {L2_BYTES / 1e6:.0f} MB L2), "
                  "no flush", "seed": a.seed}


def run_reference(args):
    """The reference arm: the FP64 oracle, as it stands, on the host cores (one thread per
    core), over a bounded sample of the workload per step (the pages ship no code)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_decode_12_gb300 import workloads as wl

    w = wl.make_workload(args.config, args.seed)
    if args.layers:
        w.layers = args.layers
    per_token = wl.kv_bytes_per_token(1, kv=args.kv)
    cores = host_cores()
    sample = oracle_samples(w, args.ref_seqs, args.seed, args.kv)
    for _ in range(args.warmup):
        oracle_run_sample(sample, args.kv, cores)
    times = []
    tokens = 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        tokens = oracle_run_sample(sample, args.kv, cores)
        times.append(time.perf_counter() - t0)
    dt = sum(times)
    value = tokens * per_token * args.steps / dt / 1e9
    desc = (f"{len(sample)} sequences of one layer per step ({tokens} KV tokens) drawn like the {w.name} workload: "
            f"append + attention for all 32 query heads, FP64 C oracle, {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(w, args, "oracle", False),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_trace(args):
    """The continuous-batching trace: the scheduler admits by page budget, prompts are
    filled into pages, and every step runs the fused decode step of all layers on the
    live batch.  value = KV bytes attended / summed device time of the decode steps;
    e2e = the same bytes / wall-clock time of the whole trace (scheduling, prefill and
    uploads included; the host schedules step s+1 while step s runs)."""
    import torch

    from paged_kv_decode_12_gb300 import pkv, workloads as wl
    from paged_kv_decode_12_gb300.trace import TraceRunner

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    steps = 500 if args.steps == 400 else args.steps
    seed = replica_seed(args.seed, rank)
    options = (VARIANTS[args.variant] | pkv.PKV_STEP_RING(args.ring) | (pkv.PKV_STEP_NO_PDL if args.no_pdl else 0)
               | (pkv.PKV_STEP_SORTED if args.sorted else 0))
    pages = args.pool_mib * 2**20 // (pkv.PKV_PAGE_BYTES_FP8 if args.kv == "fp8" else pkv.PKV_PAGE_BYTES)
    reqs = wl.trace_schedule(seed=seed, steps=steps)
    # warm-up: a short trace on a small runner (kernel attributes, tensor maps)
    warm = TraceRunner(pool_pages=4096, layers=16, max_batch=8, seed=seed + 1,
                       pages_per_chunk=args.pages_per_chunk, options=options, kv=args.kv, chains=args.chains)
    warm.run(wl.trace_schedule(seed=seed + 1, steps=max(args.warmup, 3), arrival_rate=2.0), max(args.warmup, 3))
    warm.close()
    runner = TraceRunner(pool_pages=pages, layers=16, max_batch=192, static=args.static, seed=seed,
                         pages_per_chunk=args.pages_per_chunk, options=options, kv=args.kv, chains=args.chains)
    uuid = str(getattr(torch.cuda.get_device_properties(local), "uuid", "") or "")
    sampler = ClockSampler(uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else str(local)))
    sampler.start()
    t0 = time.time()
    res = runner.run(reqs, steps)
    clocks = sampler.stop(t0, time.time())
    st, flag = pkv.pkv_check_device_error(runner.err)
    if st != pkv.PKV_OK:
        raise SystemExit(f"device error flag set during the trace: {flag:#x}")
    peak, peak_src = hbm_peak()
    gpu_s = reduce_max(res.gpu_ms / 1e3, world)
    wall_s = reduce_max(res.wall_s, world)
    value = res.kv_bytes * world / gpu_s / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * gpu_s / max(res.decode_steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.kv == "bf16" else "fp8e4m3 KV, f16 MMA, f32 softmax", "data": "synthetic",
            "config": {"workload": f"trace: {CONFIG_TEXT['trace']}", "layers": 16, "pool_mib": args.pool_mib,
                       "kv_pages": args.kv, "chains": args.chains,
                       "pages_per_chunk": args.pages_per_chunk, "ring": args.ring, "kernel_variant": args.variant,
                       "batching": "static" if args.static else "continuous", "requests": len(reqs),
                       "seed": args.seed, "l2": "KV per step far above L2 once the batch has grown; no flush"},
            "hbm_frac_of_peak": value / world / peak,
            "decode_steps_per_s_wall": res.decode_steps * world / wall_s,
            "tokens_per_s_wall": res.tokens * world / wall_s,
            "batch": {"mean": float(np.mean(res.batch_sizes)), "max": int(max(res.batch_sizes))},
            "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                         "frac": value / world / peak, "traffic": None,
                         "kernel": "fused decode step kernel, all layers of each step (events per step)",
                         "peak_source": f"{peak_src} hbm_gbs (burst copy)"},
            "e2e": {"value": res.kv_bytes * world / wall_s / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": None, "d2h_bytes_per_step": 0,
                    "path": "TraceRunner.run: scheduler, prefill, table/length uploads; the host schedules the next step while the GPU runs the current one"},
            "scheduler_stats": res.stats, "cpu_baseline": None,
            "gpu_launches": res.launches, "clocks": clocks}
    if rank == 0:
        print(json.dumps(line), flush=True)
    runner.close()
    return 0


def run_settings(args, config: str, kv: str = "bf16", path: str = "fused", split_merge: bool = False,
                 steps: int | None = None, pipelined: bool | None = None):
    """Launch settings of one measured configuration: the workload's measured defaults
    (launch table), or the command line's for the headline configuration."""
    a = argparse.Namespace(**vars(args))
    if pipelined is not None:
        a.pipelined = pipelined
    if config != args.config or kv != args.kv or path != args.path or split_merge != args.split_merge:
        a.config, a.kv, a.path, a.split_merge = config, kv, path, split_merge
        a.pages_per_chunk = DEFAULT_CHUNK[config]
        a.ring = (DEFAULT_RING if kv == "bf16" else DEFAULT_RING_FP8)[config]
        a.sorted = DEFAULT_SORTED[config] and not split_merge
        a.chains = LAUNCH.chains(config, kv, path)
        a.no_pdl = False
    if steps is not None:
        a.steps = steps
    return a


def kernel_label(a, variant_name: str) -> str:
    if a.path == "fused":
        return ("fused decode step kernel over FP8 pages (append + quantize + attention + merge)" if a.kv == "fp8"
                else f"fused decode step kernel (append + attention + merge), variant {variant_name}")
    if a.split_merge:
        return f"pkv_decode_attention two-kernel form (split kernel + LSE merge kernel), variant {variant_name}"
    return f"pkv_decode_attention kernel (attention + in-kernel LSE merge), variant {variant_name}"


def measure(a, rank, world, device, peak, peak_src, read_peak, with_cpu: bool):
    """Set up one configuration, time ``a.steps`` steps (CUDA graphs, events on the caller's
    stream), the dominant kernel per launch, the end-to-end form and (optionally) the CPU
    oracle on the same inputs.  Returns (line fields, DeviceWorkload closed)."""
    import torch

    from paged_kv_decode_12_gb300 import harness, pkv

    variant_name = a.variant
    dw = harness.setup(a.config, replica_seed(a.seed, rank), a.pages_per_chunk, VARIANTS[variant_name],
                       layers=a.layers, fused=a.path == "fused", pdl=not a.no_pdl, ring=a.ring, kv=a.kv,
                       sorted_units=a.sorted, chains=a.chains, split_merge=a.split_merge)
    w = dw.w
    cpu = cpu_baseline(dw, a.cpu_seconds, a.kv) if with_cpu else None
    harness.warm(dw, 2)
    dw.reset_q()
    ext = harness.external_events_supported()
    per_graph = max(1, min(a.steps, a.steps_per_graph))
    pipe = bool(getattr(a, "pipelined", False))
    warm_cap = harness.capture_steps(dw, max(1, min(a.warmup, per_graph)), pipelined=pipe)

    # The timed steps replay one captured graph of per_graph steps (plus one graph for the
    # remainder): a serving loop replays the same graph every step, and many distinct graph
    # instances of thousands of nodes each (micro-batch chains) cost the device time to
    # switch between.  The step time comes from these plain graphs: a timing event between
    # two launches would turn their programmatic (overlapping) dependency into a full one.
    n_full, rem = divmod(a.steps, per_graph)
    timed = [harness.capture_steps(dw, per_graph, pipelined=pipe)] * n_full
    if rem:
        timed.append(harness.capture_steps(dw, rem, pipelined=pipe))
    # per-launch durations: one instrumented graph of the same per_graph steps
    timed_ev = [harness.capture_steps(dw, per_graph, time_attention=True)] if ext else []
    torch.cuda.synchronize()

    # every timed graph is launched once before the timed region: the first launch of an
    # instantiated graph also uploads it to the device
    for cap in {id(c): c for c in timed}.values():
        cap.graph.replay()
    torch.cuda.synchronize()
    done = 0
    while done < a.warmup:
        warm_cap.graph.replay()
        done += warm_cap.steps
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    uuid = str(getattr(torch.cuda.get_device_properties(device), "uuid", "") or "")
    sampler = ClockSampler(uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else str(device.index)))
    sampler.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.time()
    start.record()
    for cap in timed:
        cap.graph.replay()
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t0, t1)
    elapsed_ms = reduce_max(start.elapsed_time(end), world, device)
    # second pass, per_graph more steps: per-launch durations of the attention kernel
    for cap in timed_ev:
        cap.graph.replay()
    torch.cuda.synchronize()

    st, flag = dw.eng.check_errors()
    if st != pkv.PKV_OK:
        raise SystemExit(f"device error flag set during the timed region: {flag:#x}")

    att_ms = [s_.elapsed_time(e_) for cap in timed_ev for (s_, e_) in cap.split_events]
    kv_step = w.kv_bytes_per_step(a.kv)
    launches = harness.attention_launches_per_step(dw)
    kv_launch = kv_step // launches  # average over the layers (and the micro-batch chains)
    steps_per_s = a.steps / (elapsed_ms / 1e3)
    value = kv_step * steps_per_s * world / 1e9
    roofline = None
    if att_ms:
        avg = sum(att_ms) / len(att_ms)
        alone = kv_launch / (avg / 1e3) / 1e9
        timing = f"external events around every attention launch in a second pass of {per_graph} steps"
        eff_ms, achieved = avg, alone
        if a.chains > 1 or a.path != "fused":
            # launches overlap on the GPU (micro-batch chains; the append kernels of the separate
            # path), and an event between two launches of one chain would serialise them: a launch's
            # GPU time comes from the timed region (step time / attention launches per step), and
            # the serialised per-launch figure is kept beside it
            eff_ms = (elapsed_ms / a.steps) / launches
            achieved = kv_launch / (eff_ms / 1e3) / 1e9
            timing = ("GPU time per attention launch = step time / attention launches per step, from the timed "
                      "region (CUDA events on the caller's stream around it)" +
                      ("; the micro-batch chains pipelined across the steps of a graph (joined once per graph, "
                       "not after every step)" if pipe else "") +
                      (", which also holds the separate path's append launches" if a.path != "fused" else "") +
                      "; launch_alone: " + timing + ", the chains one after another")
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": measured_traffic(a.config, a.path, variant_name, a.pages_per_chunk, a.ring, a.kv,
                                                a.chains, a.sorted, a.split_merge),
                    "kernel": kernel_label(a, variant_name), "timing": timing,
                    "algorithmic_bytes_per_launch": kv_launch, "avg_launch_us": eff_ms * 1e3,
                    "launches_timed": len(att_ms), "peak_source": f"{peak_src} hbm_gbs (burst copy, reads + writes)",
                    "frac_of_nominal": achieved / NOMINAL_HBM_GBS}
        if read_peak:
            roofline["frac_of_read_ceiling"] = achieved / read_peak["gbs"]
        roofline["launch_alone"] = {"achieved": alone, "frac": alone / peak, "avg_launch_us": avg * 1e3,
                                    "frac_of_read_ceiling": alone / read_peak["gbs"] if read_peak else None}

    e2e = None if a.no_e2e else measure_e2e(dw, a, world, device)
    fields = {"value": value, "unit": "GB/s", "ms_per_step": elapsed_ms / a.steps, "steps": a.steps,
              "hbm_frac_of_peak": value / world / peak,
              "hbm_frac_of_nominal": value / world / NOMINAL_HBM_GBS,
              "hbm_frac_of_read_ceiling": value / world / read_peak["gbs"] if read_peak else None,
              "steps_per_s": steps_per_s, "tokens_per_s": w.batch * steps_per_s * world,
              "attended_kv_tokens_per_s": float(w.seq_lens.sum()) * w.layers * steps_per_s * world,
              "dtype": "bf16" if a.kv == "bf16" else "fp8e4m3 KV, f16 MMA, f32 softmax",
              "config": config_block(w, a, variant_name, True), "roofline": roofline, "e2e": e2e,
              "cpu_baseline": cpu, "gpu_launches": harness.kernels_per_step(dw) * a.steps, "clocks": clocks}
    dw.eng.close()
    del dw
    torch.cuda.empty_cache()
    return fields


# further configurations measured beside the headline one in the default run: the other
# 70 %-target batch (b64), the batch-8 shape, the two named calls per layer (b64), FP8 pages,
# and b64 with its micro-batch chains pipelined across steps (DecodeEngine.steps)
EXTRA_DEFAULT = ("b64", "b8", "b64:separate", "b64:fp8", "b256:fp8", "b64:pipelined")
# extra configurations that also carry a CPU baseline on their own GPU batch: b8 its whole
# step, b64 one of its 16 layers (CPU_SAMPLE)
EXTRA_CPU = ("b64", "b8")


def parse_extra(spec: str):
    parts = spec.split(":")
    config, kv, path, split, pipelined = parts[0], "bf16", "fused", False, False
    for p in parts[1:]:
        if p == "fp8":
            kv = "fp8"
        elif p == "separate":
            path = "separate"
        elif p == "split-merge":
            path, split = "separate", True
        elif p == "pipelined":
            pipelined = True
        else:
            raise SystemExit(f"unknown extra configuration part {p!r} in {spec!r}")
    if config not in DEFAULT_CHUNK or config == "trace":
        raise SystemExit(f"unknown extra configuration {spec!r}")
    return config, kv, path, split, pipelined


def run_pkv(args):
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)

    peak, peak_src = hbm_peak()
    read_peak = None if args.no_read_ceiling else read_ceiling(device)
    head = measure(run_settings(args, args.config, args.kv, args.path, args.split_merge), rank, world, device, peak,
                   peak_src, read_peak, with_cpu=rank == 0 and world == 1 and not args.no_cpu_baseline)
    extras = {}
    specs = EXTRA_DEFAULT if args.extra == "default" else tuple(x for x in args.extra.split(",") if x and x != "none")
    for spec in specs:
        config, kv, path, split, pipelined = parse_extra(spec)
        if (config, kv, path, split, pipelined) == (args.config, args.kv, args.path, args.split_merge,
                                                    args.pipelined):
            continue
        a = run_settings(args, config, kv, path, split,
                         steps=max(args.steps, args.extra_min_steps) if config != "b256" else args.steps,
                         pipelined=pipelined)
        a.cpu_seconds = args.extra_cpu_seconds
        with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline and spec in EXTRA_CPU
        extras[spec] = measure(a, rank, world, device, peak, peak_src, read_peak, with_cpu=with_cpu)

    line = {"metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": head["config"],
            "hbm_frac_of_peak": head["hbm_frac_of_peak"], "hbm_frac_of_nominal": head["hbm_frac_of_nominal"],
            "hbm_frac_of_read_ceiling": head["hbm_frac_of_read_ceiling"],
            "steps_per_s": head["steps_per_s"], "tokens_per_s": head["tokens_per_s"],
            "attended_kv_tokens_per_s": head["attended_kv_tokens_per_s"],
            "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
            "read_ceiling": read_peak, "nominal_hbm_gbs": NOMINAL_HBM_GBS,
            "configs": extras}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def measure_e2e(dw, args, world, device):
    """Same metric through DecodeEngine.run_host_steps: every step copies q, k_new, v_new,
    positions and lengths (packed, one copy) from pinned host memory and its output back,
    through rotating buffers on two copy streams, so that the copies of the neighbouring
    steps overlap the step's compute.  Each step's kernels replay a captured graph of that
    step (one graph per buffer); the copies are stream operations between the replays."""
    import torch

    from paged_kv_decode_12_gb300 import harness

    io = harness.host_pinned_inputs(dw)
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    group = max(1, args.e2e_group)
    nbuf = max(2 * group, -(-args.e2e_buffers // group) * group)
    outs = [dw.out] + [torch.empty_like(dw.out) for _ in range(nbuf - 1)]
    n = max(group, args.e2e_steps // group * group)
    dw.eng.run_host_steps(io, outs, out_host, len(outs))   # eager first pass: every buffer once
    torch.cuda.synchronize()
    graphs = dw.eng.step_graphs(io, outs, group, pipelined=bool(getattr(args, "pipelined", False)))
    dw.eng.run_host_steps(io, outs, out_host, len(outs), graphs=graphs, group=group)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    dw.eng.run_host_steps(io, outs, out_host, n, graphs=graphs, group=group)
    end.record()
    torch.cuda.synchronize()
    ms = reduce_max(start.elapsed_time(end), world, device)
    h2d = io.bytes
    d2h = out_host.numel() * out_host.element_size()
    return {"value": dw.w.kv_bytes_per_step(dw.eng.kv) * n * world / (ms / 1e3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms / n,
            "path": "DecodeEngine.run_host_steps (per step: one H2D copy of the packed pinned inputs and one D2H "
                    f"copy of the output, through {len(outs)} rotating buffers on two copy streams so that they "
                    f"overlap the neighbouring steps' compute; the steps' kernels replay captured graphs of {group} "
                    "steps" + (" with the micro-batch chains pipelined across them" if getattr(args, "pipelined", False)
                               else "") +
                    ", the copies are stream operations between the replays)", "steps_per_graph": group}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--config", choices=sorted(CONFIG_TEXT), default="b256")
    ap.add_argument("--pages-per-chunk", type=int, default=None,
                    help="pages per work unit (default: the measured best for the workload, "
                         + ", ".join(f"{k} {v}" for k, v in DEFAULT_CHUNK.items()) + ")")
    ap.add_argument("--variant", choices=sorted(VARIANTS), default="default")
    ap.add_argument("--path", choices=["fused", "separate"], default="fused",
                    help="one fused kernel per layer, or pkv_append_rope + pkv_decode_attention launches")
    ap.add_argument("--split-merge", action="store_true",
                    help="separate path: the two-kernel attention form (split kernel + LSE merge kernel)")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--sorted", action="store_true", default=None,
                    help="grid schedule: dispatch work units largest first (PKV_STEP_SORTED; default: per workload, "
                         + ", ".join(f"{k} {v}" for k, v in DEFAULT_SORTED.items()) + ")")
    ap.add_argument("--unsorted", action="store_true", help="grid schedule: dispatch units in grid order")
    ap.add_argument("--pool-mib", type=int, default=16384, help="trace: KV pool size (the engine's default is 128)")
    ap.add_argument("--static", action="store_true", help="trace: static batching instead of continuous")
    ap.add_argument("--ring", type=int, default=None, choices=[2, 3, 4],
                    help="grid schedule: TMA stages per warp (default: the measured best for the workload)")
    ap.add_argument("--chains", type=int, default=None,
                    help="fused path: micro-batch chains, each a per-layer launch chain over a contiguous row "
                         "group on its own stream (default: per workload, BF16 "
                         + ", ".join(f"{k} {v}" for k, v in DEFAULT_CHAINS.items()) + "; FP8 "
                         + ", ".join(f"{k} {v}" for k, v in DEFAULT_CHAINS_FP8.items()) + ")")
    ap.add_argument("--pipelined", action="store_true",
                    help="micro-batch chains pipelined across the steps of a captured graph "
                         "(DecodeEngine.steps: joined once per graph instead of after every step)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="KV page format: BF16 (the engine's) or FP8 E4M3 with per-row scales")
    ap.add_argument("--seed", type=int, default=12)
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (small profiling runs)")
    ap.add_argument("--steps-per-graph", type=int, default=25)
    ap.add_argument("--e2e-steps", type=int, default=400,
                    help="end-to-end steps timed (the first group's uploads and the last group's copies back "
                         "are not overlapped: more steps measure the steady state)")
    ap.add_argument("--e2e-buffers", type=int, default=2, help="end-to-end input/output buffers in rotation "
                    "(at least twice --e2e-group)")
    ap.add_argument("--e2e-group", type=int, default=8, help="end-to-end steps per captured graph replay")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="CPU baseline: seconds of oracle work, half single-threaded, half on every host core")
    ap.add_argument("--extra-cpu-seconds", type=float, default=4.0,
                    help="CPU baseline of the extra configurations " + ", ".join(EXTRA_CPU) + ": seconds of oracle "
                         "work each")
    ap.add_argument("--ref-seqs", type=int, default=16, help="sequences per reference-arm step")
    ap.add_argument("--extra", default="default",
                    help="further configurations measured in the same run and reported under 'configs': "
                         "comma-separated workload[:fp8][:separate|:split-merge] items, 'none', or 'default' ("
                         + ", ".join(EXTRA_DEFAULT) + ")")
    ap.add_argument("--extra-min-steps", type=int, default=200, help="at least this many timed steps per extra "
                    "configuration other than b256")
    ap.add_argument("--no-read-ceiling", action="store_true", help="skip the read-only HBM probe")
    args = ap.parse_args(argv)
    if args.pages_per_chunk is None:
        args.pages_per_chunk = DEFAULT_CHUNK[args.config]
    if args.ring is None:
        args.ring = DEFAULT_RING[args.config] if args.kv == "bf16" else DEFAULT_RING_FP8[args.config]
    if args.sorted is None:
        args.sorted = DEFAULT_SORTED[args.config] and not args.unsorted and not args.split_merge
    elif args.unsorted:
        raise SystemExit("--sorted and --unsorted exclude each other")
    if args.split_merge and args.path != "separate":
        raise SystemExit("--split-merge selects the separate path's two-kernel attention (--path separate)")
    if args.chains is None:
        args.chains = LAUNCH.chains(args.config, args.kv, args.path)
    if args.impl == "reference":
        return run_reference(args)
    if args.config == "trace":
        return run_trace(args)
    return run_pkv(args)


if __name__ == "__main__":
    sys.exit(main())
