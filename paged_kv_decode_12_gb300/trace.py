"""Continuous-batching trace over the C ABI: scheduler, prefill page fill, decode steps.

Each step of the trace: submit the requests arriving at this step, admit waiting
requests by page budget (``pkv_sched_admit``; FIFO, rejection, lazy pages), fill
each admitted prompt's pages one prompt at a time (``pkv_prefill_append``; the
README summary's "prefill fills the prompt's pages", prompts between decode
iterations), then build the decode batch (``pkv_sched_decode_batch``: one new token
per active sequence, pages taken at page boundaries) and run the fused decode step
for every layer (``pkv_decode_step``).  Activations are seeded synthetic draws:
there is no model, so prompt K/V, q, k_new and v_new are N(0,1) BF16 (the attention
path does not depend on their origin).

PyTorch allocates device memory and provides the stream; the scheduler is native
(C++ in libpkv) and every step of the computation runs in libpkv's kernels.
"""
from __future__ import annotations

import dataclasses
import math
import time

import numpy as np
import torch

from . import pkv
from . import workloads as wl


@dataclasses.dataclass
class TraceResult:
    steps: int
    decode_steps: int              # steps with a non-empty batch
    gpu_ms: float                  # summed device time of the decode steps (events)
    wall_s: float                  # whole trace, host scheduling and uploads included
    kv_bytes: int                  # K/V bytes attended over the trace
    tokens: int                    # decode tokens produced (one per active sequence per step)
    batch_sizes: list
    stats: dict
    launches: int = 0              # library kernel launches (decode steps of every layer and chain, prefills)


class TraceRunner:
    def __init__(self, pool_pages: int, layers: int = 16, max_batch: int = 192, max_blocks: int = wl.MAX_BLOCKS,
                 max_context: int = wl.MAX_CONTEXT, static: bool = False, seed: int = wl.DEFAULT_SEED,
                 pages_per_chunk: int = 32, options: int = pkv.PKV_STEP_RING(2), device: str = "cuda",
                 kv: str = "bf16", chains: int = 1):
        self.device = torch.device(device)
        self.layers, self.max_batch, self.max_blocks, self.max_context = layers, max_batch, max_blocks, max_context
        self.pages_per_chunk, self.options, self.seed = pages_per_chunk, options, seed
        self.scale = 1.0 / math.sqrt(wl.HEAD_DIM)
        self.kv = kv
        self.page_bytes = pkv.PKV_PAGE_BYTES_FP8 if kv == "fp8" else pkv.PKV_PAGE_BYTES
        self.slab = torch.zeros(pool_pages * self.page_bytes, dtype=torch.uint8, device=self.device)
        if kv == "fp8":  # prompts are quantized by the prefill, decode tokens by the step
            self.pool = pkv.pkv_pool_create_fp8(self.slab, self.slab.numel(), seed=seed)
        else:
            self.pool = pkv.pkv_pool_create(self.slab, self.slab.numel(), seed=seed)
        self.num_pages = pool_pages
        self.sched = pkv.pkv_sched_create(self.pool, layers, max_blocks, max_context, max_batch,
                                          pkv.PKV_SCHED_STATIC if static else pkv.PKV_SCHED_CONTINUOUS)
        self.rope = pkv.rope_table(max_context, self.device, wl.ROPE_THETA)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.ws_bytes = pkv.pkv_decode_step_workspace_bytes(max_batch, max_blocks, pages_per_chunk)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
        # micro-batch chains (see engine.chain_bounds): per chain a stream and a workspace
        if chains < 1:
            raise ValueError(f"chains must be >= 1, not {chains}")
        self.chains = chains
        self.chain_streams = [torch.cuda.Stream(device=self.device) for _ in range(chains)] if chains > 1 else []
        self.chain_ws = [torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
                         for _ in range(chains)] if chains > 1 else []

        def draw(shape, s):
            return wl.fill_bf16_normal_(torch.empty(shape, dtype=torch.bfloat16, device=self.device), s)

        # q is rotated in place by every step: each step starts from the unrotated draw q0,
        # as a real step starts from freshly projected queries
        self.q0 = draw((layers, max_batch, wl.NUM_Q_HEADS, wl.HEAD_DIM), seed + 1)
        self.q = self.q0.clone()
        self.k_new = draw((layers, max_batch, wl.NUM_KV_HEADS, wl.HEAD_DIM), seed + 2)
        self.v_new = draw((layers, max_batch, wl.NUM_KV_HEADS, wl.HEAD_DIM), seed + 3)
        self.out = torch.zeros((layers, max_batch, wl.NUM_Q_HEADS, wl.HEAD_DIM), dtype=torch.bfloat16,
                               device=self.device)
        # block tables of a decode step, compact [layers][B][max_blocks] (layer stride B x max_blocks)
        self.bt = torch.full((layers * max_batch * max_blocks,), -1, dtype=torch.int32, device=self.device)
        self.lens = torch.zeros(max_batch, dtype=torch.int32, device=self.device)
        self.prompt_bt = torch.full((max_batch, layers, max_blocks), -1, dtype=torch.int32, device=self.device)
        # two sets of pinned host buffers that the scheduler writes into directly and that are
        # copied to the device asynchronously; a set is rewritten only after the copies out of
        # it have finished (its event), so the host schedules a step while earlier ones run
        def pinned(n, dtype):
            return torch.empty(n, dtype=dtype).pin_memory()

        self._stage = [dict(ids=np.empty(max_batch, np.int64), lens=pinned(max_batch, torch.int32),
                            bt=pinned(layers * max_batch * max_blocks, torch.int32),
                            pids=np.empty(max_batch, np.int64), plens=np.empty(max_batch, np.int32),
                            pbt=pinned(max_batch * layers * max_blocks, torch.int32), ev=None) for _ in range(2)]
        self._nstage = 0
        self.launches = 0
        # every decode call gets its arguments as addresses computed from these bases and row
        # strides (no tensor views per call: the trace launches from the host every step)
        kv_row, q_row = wl.NUM_KV_HEADS * wl.HEAD_DIM * 2, wl.NUM_Q_HEADS * wl.HEAD_DIM * 2
        self._base = dict(k=self.k_new.data_ptr(), v=self.v_new.data_ptr(), q=self.q.data_ptr(),
                          bt=self.bt.data_ptr(), lens=self.lens.data_ptr(), out=self.out.data_ptr(),
                          rope=self.rope.data_ptr(), err=self.err.data_ptr())
        self._stride = dict(kv=kv_row, q=q_row, bt=max_blocks * 4)
        self._fork = torch.cuda.Event() if chains > 1 else None
        self._joins = [torch.cuda.Event() for _ in range(chains)] if chains > 1 else []
        self._prompt_seed = seed + 100
        self.prompt_seeds = {}  # request id -> (seed of its prompt K/V draw, prompt length)

    def close(self):
        if self.sched is not None:
            pkv.pkv_sched_destroy(self.sched)
            self.sched = None
        if self.pool is not None:
            pkv.pkv_pool_destroy(self.pool)
            self.pool = None

    # ------------------------------------------------------------------ pieces
    def prompt_kv(self, seed: int, prompt_len: int):
        """The seeded N(0,1) prompt K and V of every layer, [layers][prompt_len][8][64] BF16."""
        g = torch.Generator(device=self.device)
        g.manual_seed(seed)
        shape = (self.layers, prompt_len, wl.NUM_KV_HEADS, wl.HEAD_DIM)
        k = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32).to(torch.bfloat16)
        v = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32).to(torch.bfloat16)
        return k, v

    def prefill(self, bt_rows, prompt_len: int, rid: int = -1, slot: int = 0):
        """Fill one prompt's pages in every layer with seeded N(0,1) K/V.  ``bt_rows``
        [layers][max_blocks]: a device tensor (row ``slot`` of the prompt tables, already
        uploaded) or host rows (copied to that row first)."""
        rows = self.prompt_bt[slot]
        if not isinstance(bt_rows, torch.Tensor) or not bt_rows.is_cuda:
            rows.copy_(torch.as_tensor(np.asarray(bt_rows)))
        self._prompt_seed += 1
        self.prompt_seeds[rid] = (self._prompt_seed, prompt_len)
        k, v = self.prompt_kv(self._prompt_seed, prompt_len)
        pkv.pkv_prefill_append(self.pool, k, v, rows, self.max_blocks, self.layers, 0, prompt_len, self.rope,
                               self.max_context, self.err)
        self.launches += 1

    def _layers(self, r0: int, r1: int, B: int, ws, stream=None):
        """Every layer of one decode step for batch rows r0..r1-1 of B (contiguous slices of
        the per-layer [max_batch] arrays and of the compact [layers][B] tables, as addresses)."""
        self.launches += self.layers
        a, st = self._base, self._stride
        ws_ptr, lens = ws.data_ptr(), a["lens"] + 4 * r0
        stream = torch.cuda.current_stream(self.device).cuda_stream if stream is None else stream.cuda_stream
        # one library call for all layers: layer l's rows are r0.. of layer l's arrays
        pkv.pkv_decode_step_layers(self.pool, self.layers, a["k"] + r0 * st["kv"], a["v"] + r0 * st["kv"],
                                   a["q"] + r0 * st["q"], a["bt"] + r0 * st["bt"], self.max_blocks, lens, r1 - r0,
                                   a["rope"], self.max_context, self.scale, self.pages_per_chunk, ws_ptr,
                                   self.ws_bytes, a["out"] + r0 * st["q"], a["err"], stream, self.options,
                                   self.max_batch * st["kv"] // 2, self.max_batch * st["q"] // 2,
                                   B * st["bt"] // 4)

    def decode(self, B: int, lens_host=None):
        """All layers of one decode step over the first B batch rows (tables: compact
        [layers][B][max_blocks]); with chains, as micro-batch chains cut by the rows' page
        counts (``lens_host``)."""
        k = min(self.chains, B)
        if k <= 1:
            self._layers(0, B, B, self.ws)
            return
        from .engine import chain_bounds

        bounds = chain_bounds(B, k, lens_host)
        cur = torch.cuda.current_stream(self.device)
        self._fork.record(cur)
        for i in range(k):
            s = self.chain_streams[i]
            s.wait_event(self._fork)
            self._layers(bounds[i], bounds[i + 1], B, self.chain_ws[i], s)
            self._joins[i].record(s)
        for i in range(k):
            cur.wait_event(self._joins[i])

    # ------------------------------------------------------------------ trace
    def run(self, requests, steps: int, before_step=None, after_step=None) -> TraceResult:
        """Run ``steps`` trace steps.  ``before_step(step, ids, lens, bt_host)`` and
        ``after_step(step, ids, lens, bt_host)`` (optional) see each decode batch."""
        by_step = {}
        for r in requests:
            by_step.setdefault(r.arrival_step, []).append(r)
        gpu_ms, kv_bytes, tokens, decode_steps, sizes = 0.0, 0, 0, 0, []
        timed = []
        self.launches = 0
        per_token = wl.kv_bytes_per_token(self.layers, kv=self.kv)
        row = self.layers * self.max_blocks
        t0 = time.perf_counter()
        for step in range(steps):
            for r in by_step.get(step, []):
                try:
                    pkv.pkv_sched_submit(self.sched, r.rid, r.prompt_len, r.max_new)
                except pkv.PkvError as e:
                    if e.status != pkv.PKV_ERR_BUDGET_EXCEEDS_POOL:
                        raise
            st = self._stage[self._nstage % 2]
            self._nstage += 1
            if st["ev"] is not None:
                st["ev"].synchronize()  # the copies out of this set (two steps ago) are done
            ids, plens, bt_rows = pkv.pkv_sched_admit(self.sched, self.max_batch, self.layers, self.max_blocks,
                                                      st["pids"], st["plens"], st["pbt"].numpy())
            if ids.size:
                self.prompt_bt.view(-1)[: ids.size * row].copy_(st["pbt"][: ids.size * row], non_blocking=True)
            for i in range(ids.size):
                self.prefill(self.prompt_bt[i], int(plens[i]), int(ids[i]), i)
            ids, lens, bt = pkv.pkv_sched_decode_batch(self.sched, self.max_batch, self.layers, self.max_blocks,
                                                       st["ids"], st["lens"].numpy(), st["bt"].numpy())
            B = ids.size
            sizes.append(B)
            if B:
                self.lens[:B].copy_(st["lens"][:B], non_blocking=True)
                self.bt[: B * row].copy_(st["bt"][: B * row], non_blocking=True)
            st["ev"] = torch.cuda.Event()
            st["ev"].record()  # after every copy out of this set (prompt tables included)
            if B == 0:
                continue
            self.q[:, :B].copy_(self.q0[:, :B])
            if before_step or after_step:   # the callbacks keep what they see: copies
                ids, lens, bt = ids.copy(), lens.copy(), bt.copy()
            if before_step:
                before_step(step, ids, lens, bt)
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record()
            self.decode(B, lens)
            end.record()
            if after_step:
                after_step(step, ids, lens, bt)
            # the events are read after the trace: the host schedules the next step while
            # this one runs (every device-side use of a buffer is ordered on the stream)
            timed.append((start, end))
            kv_bytes += int(lens.astype(np.int64).sum()) * per_token
            tokens += B
            decode_steps += 1
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        gpu_ms = sum(a.elapsed_time(b) for a, b in timed)
        return TraceResult(steps, decode_steps, gpu_ms, wall, kv_bytes, tokens, sizes,
                           pkv.pkv_sched_get_stats(self.sched), self.launches)
