"""Device-side set-up of a named workload and CUDA-graph capture of decode steps.

Shared by ``bench.py`` and the GPU tests so that the tests check exactly the
launch configuration the benchmark times.  Inputs are seeded synthetic draws
(see ``workloads``); nothing here computes any part of the method.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import pkv
from . import workloads as wl
from .engine import DecodeEngine


@dataclasses.dataclass
class DeviceWorkload:
    w: wl.Workload
    eng: DecodeEngine
    q: torch.Tensor        # [layers][B][32][64] bf16 (rotated in place by each step's append)
    q0: torch.Tensor       # the unrotated draw, kept for reference checks
    k_new: torch.Tensor    # [layers][B][8][64] bf16
    v_new: torch.Tensor
    pos: torch.Tensor      # [B] int32
    seq_lens: torch.Tensor # [B] int32
    out: torch.Tensor      # [layers][B][32][64] bf16

    def step(self, stream=None, layer_hook=None):
        self.eng.step(self.q, self.k_new, self.v_new, self.pos, self.seq_lens, self.out, stream, layer_hook)

    def reset_q(self):
        self.q.copy_(self.q0)


def setup(name: str, seed: int = wl.DEFAULT_SEED, pages_per_chunk: int = 16,
          variant: int = pkv.PKV_DECODE_DEFAULT, layers: int | None = None, device: str = "cuda",
          fused: bool = True, pdl: bool = True, ring: int = 0, kv: str = "bf16", sorted_units: bool = False,
          chains: int = 1, split_merge: bool = False) -> DeviceWorkload:
    """Build the named workload on the GPU: pool filled with N(0,1) BF16 (plus the
    key outliers of ``b64``) or, with ``kv="fp8"``, with FP8 pages drawn by
    ``workloads.fill_fp8_pages_``; block tables from the library's seeded
    allocator, per-layer q / k_new / v_new draws, positions = lengths - 1.
    ``chains`` > 1 runs the step as that many micro-batch chains (see engine); ``fused=False``
    runs pkv_append_rope + pkv_decode_attention per layer (``split_merge``: the two-kernel
    attention form)."""
    w = wl.make_workload(name, seed)
    if layers is not None and layers != w.layers:
        w = dataclasses.replace(w, layers=layers, pool_pages=w.pool_pages * layers // w.layers)
    eng = DecodeEngine(w.pool_pages, w.layers, w.batch, w.max_blocks, pages_per_chunk, variant, pool_seed=seed,
                       device=device, fused=fused, pdl=pdl, ring=ring, kv=kv, sorted_units=sorted_units,
                       chains=chains, split_merge=split_merge)
    if kv == "fp8":
        codes, scales = eng.fp8_views()
        wl.fill_fp8_pages_(codes, scales, seed, w.key_outlier_frac)
    else:
        pool = eng.pool_view()
        wl.fill_bf16_normal_(pool, seed)
        wl.scale_key_rows_(pool, w.key_outlier_frac, seed + 7)
    eng.build_tables(w.seq_lens)
    dev = eng.device

    def draw(shape, s):
        t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        return wl.fill_bf16_normal_(t, s)

    L, B = w.layers, w.batch
    q0 = draw((L, B, wl.NUM_Q_HEADS, wl.HEAD_DIM), seed + 1)
    k_new = draw((L, B, wl.NUM_KV_HEADS, wl.HEAD_DIM), seed + 2)
    v_new = draw((L, B, wl.NUM_KV_HEADS, wl.HEAD_DIM), seed + 3)
    pos = torch.from_numpy(w.positions).to(dev)
    seq_lens = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.zeros((L, B, wl.NUM_Q_HEADS, wl.HEAD_DIM), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize(dev)
    return DeviceWorkload(w, eng, q0.clone(), q0, k_new, v_new, pos, seq_lens, out)


def kernels_per_step(dw: DeviceWorkload) -> int:
    """Library kernel launches in one step, per layer and micro-batch chain: one fused
    kernel (BF16 or FP8 pages), or (separate path) the append and the attention kernel
    (two-kernel form: the split kernel and, when a sequence can span several chunks,
    the merge kernel)."""
    per_layer = 1
    if not dw.eng.fused:
        two_kernel = bool(dw.eng.attn_options & pkv.PKV_DECODE_SPLIT_MERGE)
        multi = (dw.w.max_blocks + dw.eng.pages_per_chunk - 1) // dw.eng.pages_per_chunk > 1
        per_layer = 2 + (1 if two_kernel and multi else 0)
    return dw.w.layers * dw.eng.chains * per_layer


def attention_launches_per_step(dw: DeviceWorkload) -> int:
    """Attention launches (the dominant kernel) in one step: one per layer and chain."""
    return dw.w.layers * dw.eng.chains


def external_events_supported() -> bool:
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


@dataclasses.dataclass
class CapturedSteps:
    graph: torch.cuda.CUDAGraph
    steps: int
    split_events: list  # (start, end) event pairs around each attention launch, or []


def capture_steps(dw: DeviceWorkload, steps: int, time_attention: bool = False,
                  pipelined: bool = False) -> CapturedSteps:
    """Capture ``steps`` consecutive decode steps into one CUDA graph.  With
    ``time_attention`` an external timing event is recorded before and after every
    attention launch inside the graph (each graph has its own events).  ``pipelined``:
    the steps through ``DecodeEngine.steps`` (micro-batch chains joined once, after the
    last step)."""
    events = []

    def hook(layer, phase):
        if phase == "before":
            events.append([torch.cuda.Event(enable_timing=True, external=True), None])
            events[-1][0].record()
        else:
            events[-1][1] = torch.cuda.Event(enable_timing=True, external=True)
            events[-1][1].record()

    if pipelined and time_attention:
        raise ValueError("per-launch events need the steps one after another")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if pipelined:
            dw.eng.steps([(dw.q, dw.k_new, dw.v_new, dw.pos, dw.seq_lens, dw.out)] * steps)
        else:
            for _ in range(steps):
                dw.step(layer_hook=hook if time_attention else None)
    return CapturedSteps(g, steps, [tuple(e) for e in events])


def warm(dw: DeviceWorkload, n: int = 2) -> None:
    """Eager steps on a side stream (sets kernel attributes, encodes the tensor map)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(n):
            dw.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()


def host_pinned_inputs(dw: DeviceWorkload):
    """One step's inputs (the unrotated q, k_new, v_new, pos, seq_lens) packed in pinned host
    memory, with a device buffer of the same layout (for the end-to-end measurement)."""
    from .engine import PackedIO

    return PackedIO({"q": dw.q0, "k_new": dw.k_new, "v_new": dw.v_new, "pos": dw.pos, "seq_lens": dw.seq_lens},
                    dw.eng.device)


def sample_units(w: wl.Workload, n: int, seed: int) -> list:
    """Seeded (layer, sequence, query head) samples, always including the last
    sequence, the first, and a sequence at each boundary length present."""
    rng = np.random.default_rng(seed)
    picks = {(0, 0, 0), (w.layers - 1, w.batch - 1, wl.NUM_Q_HEADS - 1)}
    for b, L in enumerate(w.seq_lens):
        if int(L) in (1, 16, 17, 32, 33, 2048) and len(picks) < n // 2:
            picks.add((int(rng.integers(w.layers)), b, int(rng.integers(wl.NUM_Q_HEADS))))
    while len(picks) < n:
        picks.add((int(rng.integers(w.layers)), int(rng.integers(w.batch)), int(rng.integers(wl.NUM_Q_HEADS))))
    return sorted(picks)
