"""Multi-layer decode step over the C ABI: the public entry point a user calls.

``DecodeEngine`` owns the device buffers one decode step needs (the KV page
slab, per-layer block tables, the RoPE factor table, the attention workspace
and the device error flag) and runs, for every layer, the two library calls of
the hot path: ``pkv_append_rope`` (RoPE + page-slot append of the new token,
query rotated in place) then ``pkv_decode_attention`` (paged GQA attention over
the sequence's pages).  PyTorch only allocates memory and provides the stream;
every step of the computation runs in libpkv's kernels.

``run_host`` is the end-to-end form: inputs come from pinned host memory and
the result goes back to it, with the copies on the same stream as the kernels.

By default each layer runs as one fused launch (``pkv_decode_step``: append and
attention in one kernel); ``fused=False`` runs the two named calls instead.

Micro-batch chains (``chains=K``): the batch rows are cut into K contiguous
groups, each group runs its own chain of per-layer launches on its own stream
(forked from and joined back to the caller's stream), so one group's layer tail
overlaps another group's streaming.  Layer order is kept inside every group;
sequences never interact, so every output byte is the same as with one chain.

``steps()`` runs several decode steps with the chains pipelined across the step
boundaries: every chain runs its rows through step 0, 1, ... back to back and the
chains are joined once, after the last step, instead of after every step.  Every
step still appends one token to every sequence and attends over all of its pages;
only the barrier that made all micro-batches finish step s before any began step
s + 1 is gone (a micro-batch's next step depends on its own sequences only).  The
bytes written are those of the same steps run one by one.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import pkv
from . import workloads as wl


class DecodeEngine:
    def __init__(self, num_pages: int, layers: int, batch: int, max_blocks: int = wl.MAX_BLOCKS,
                 pages_per_chunk: int = 16, variant: int = pkv.PKV_DECODE_DEFAULT, max_pos: int = wl.MAX_CONTEXT,
                 theta: float = wl.ROPE_THETA, pool_seed: int = 0, device: str = "cuda", fused: bool = True,
                 pdl: bool = True, ring: int = 0, kv: str = "bf16", sorted_units: bool = False, chains: int = 1,
                 split_merge: bool = False):
        if kv not in ("bf16", "fp8"):
            raise ValueError(f"kv must be 'bf16' or 'fp8', not {kv!r}")
        if not 1 <= chains <= batch:
            raise ValueError(f"chains must be in [1, batch], not {chains}")
        if split_merge and fused:
            raise ValueError("split_merge selects the two-kernel attention of the separate path (fused=False)")
        self.kv = kv
        self.device = torch.device(device)
        self.layers, self.batch, self.max_blocks = layers, batch, max_blocks
        self.pages_per_chunk, self.variant, self.max_pos = pages_per_chunk, variant, max_pos
        self.scale = 1.0 / math.sqrt(wl.HEAD_DIM)
        self.page_bytes = pkv.PKV_PAGE_BYTES_FP8 if kv == "fp8" else pkv.PKV_PAGE_BYTES
        self.slab = torch.empty(num_pages * self.page_bytes, dtype=torch.uint8, device=self.device)
        if kv == "fp8":
            self.pool = pkv.pkv_pool_create_fp8(self.slab, self.slab.numel(), seed=pool_seed)
        else:
            self.pool = pkv.pkv_pool_create(self.slab, self.slab.numel(), seed=pool_seed)
        self.num_pages = num_pages
        self.rope = pkv.rope_table(max_pos, self.device, theta)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        # the attention workspace (the fused step's too) starts with per-(sequence, KV head)
        # merge counters that must be zero before the first call (every call leaves them zero)
        self.ws_bytes = pkv.pkv_decode_workspace_bytes(batch, max_blocks, pages_per_chunk)
        self.workspace = torch.zeros(max(self.ws_bytes, 16), dtype=torch.uint8, device=self.device)
        self.step_ws_bytes = pkv.pkv_decode_step_workspace_bytes(batch, max_blocks, pages_per_chunk)
        self.step_ws = self.workspace
        self.fused = fused
        # launch options of the fused step and of the separate path's attention call
        self.step_options = (variant | (0 if pdl else pkv.PKV_STEP_NO_PDL) | pkv.PKV_STEP_RING(ring)
                             | (pkv.PKV_STEP_SORTED if sorted_units else 0))
        self.attn_options = pkv.PKV_DECODE_SPLIT_MERGE | variant if split_merge else self.step_options
        self.bt = None
        self.bt_host = None
        self.chains = chains
        self.chain_bounds = chain_bounds(batch, chains)
        # each chain has its own stream and its own workspace (counters start at zero)
        self.chain_streams = [torch.cuda.Stream(device=self.device) for _ in range(chains)] if chains > 1 else []
        self.chain_ws = [torch.zeros(self.step_ws_bytes, dtype=torch.uint8, device=self.device)
                         for _ in range(chains)] if chains > 1 else []

    # ------------------------------------------------------------------ setup
    def pool_view(self) -> torch.Tensor:
        """The slab as BF16 [pages][2 (K, V)][8 KV heads][16 slots][64 dims] (BF16 pools)."""
        if self.kv != "bf16":
            raise ValueError("pool_view is the BF16 layout; use fp8_views for an FP8 pool")
        return self.slab.view(torch.bfloat16).view(self.num_pages, 2, wl.NUM_KV_HEADS, wl.PAGE_SIZE,
                                                   wl.HEAD_DIM)

    def fp8_views(self):
        """(codes uint8 [pages][2][8][16 x 64 bytes], scales float32 [pages][2][8][16]) of an FP8
        pool; the code bytes are in storage order (K rows; V codes interleaved by token pair)."""
        if self.kv != "fp8":
            raise ValueError("fp8_views needs an FP8 pool")
        # a page is one 2176-byte unit per KV head: codes [2][16][64], then scales [2][16]
        H, P, D = wl.NUM_KV_HEADS, wl.PAGE_SIZE, wl.HEAD_DIM
        units = self.slab.view(self.num_pages, H, self.page_bytes // H)
        codes = units[:, :, :2 * P * D].view(self.num_pages, H, 2, P, D).permute(0, 2, 1, 3, 4)
        scales = units[:, :, 2 * P * D:].view(torch.float32).view(self.num_pages, H, 2, P).permute(0, 2, 1, 3)
        return codes, scales

    def build_tables(self, seq_lens) -> np.ndarray:
        """Allocate pages for every (layer, sequence) and upload the block tables; the
        micro-batch chains (if any) are cut to balance their pages."""
        bt = pkv.pkv_block_tables_build(self.pool, self.layers, seq_lens, self.max_blocks)
        self.set_tables(bt)
        self.chain_bounds = chain_bounds(self.batch, self.chains, seq_lens)
        return bt

    def set_tables(self, bt_host: np.ndarray) -> None:
        assert bt_host.shape == (self.layers, self.batch, self.max_blocks)
        self.bt_host = np.ascontiguousarray(bt_host, dtype=np.int32)
        self.bt = torch.from_numpy(self.bt_host).to(self.device)

    def close(self) -> None:
        if self.pool is not None:
            pkv.pkv_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ step
    def append(self, layer: int, k_new, v_new, q, pos_dev, stream=None, rows=None) -> None:
        """pkv_append_rope of one layer (rows r0..r1-1 with ``rows=(r0, r1)``)."""
        r0, r1 = rows if rows is not None else (0, self.batch)
        pkv.pkv_append_rope(self.pool, k_new[r0:r1], v_new[r0:r1], q[r0:r1], self.bt[layer, r0:r1], self.max_blocks,
                            pos_dev[r0:r1], r1 - r0, self.rope, self.max_pos, self.err, stream)

    def attention(self, layer: int, q, seq_lens_dev, out, stream=None, variant=None, rows=None,
                  workspace=None) -> None:
        """pkv_decode_attention(_variant) of one layer with the engine's attention options
        (or ``variant``); rows and workspace as for ``fused_layer``."""
        r0, r1 = rows if rows is not None else (0, self.batch)
        pkv.pkv_decode_attention_variant(self.pool, q[r0:r1], self.bt[layer, r0:r1], self.max_blocks,
                                         seq_lens_dev[r0:r1], r1 - r0, self.scale, self.pages_per_chunk,
                                         self.workspace if workspace is None else workspace, self.ws_bytes,
                                         out[r0:r1], self.err, stream,
                                         self.attn_options if variant is None else variant)

    def fused_layer(self, layer: int, q, k_new, v_new, seq_lens_dev, out, stream=None, rows=None,
                    workspace=None) -> None:
        """Append + attention of one layer in one launch (positions are seq_lens - 1); with
        ``rows=(r0, r1)`` for the batch rows r0..r1-1 only (contiguous slices of every argument)."""
        r0, r1 = rows if rows is not None else (0, self.batch)
        pkv.pkv_decode_step(self.pool, k_new[r0:r1], v_new[r0:r1], q[r0:r1], self.bt[layer, r0:r1], self.max_blocks,
                            seq_lens_dev[r0:r1], r1 - r0, self.rope, self.max_pos, self.scale, self.pages_per_chunk,
                            self.step_ws if workspace is None else workspace, self.step_ws_bytes, out[r0:r1],
                            self.err, stream, self.step_options)

    def fused_layers(self, q, k_new, v_new, seq_lens_dev, out, stream=None, rows=None, workspace=None) -> None:
        """Every layer's fused launch for batch rows ``rows`` (default: all) in one library
        call (``pkv_decode_step_layers``): q, k_new, v_new, out are [layers][B][...] with
        contiguous rows; a layer's arrays are the layer-0 rows plus the tensors' layer stride."""
        r0, r1 = rows if rows is not None else (0, self.batch)
        ws = self.step_ws if workspace is None else workspace
        if k_new.stride(0) != v_new.stride(0) or q.stride(0) != out.stride(0):
            for layer in range(self.layers):  # layer strides the one call cannot express
                self.fused_layer(layer, q[layer], k_new[layer], v_new[layer], seq_lens_dev, out[layer], stream,
                                 rows, ws)
            return
        pkv.pkv_decode_step_layers(self.pool, self.layers, k_new[0, r0:r1], v_new[0, r0:r1], q[0, r0:r1],
                                   self.bt[0, r0:r1], self.max_blocks, seq_lens_dev[r0:r1], r1 - r0, self.rope,
                                   self.max_pos, self.scale, self.pages_per_chunk, ws, self.step_ws_bytes,
                                   out[0, r0:r1], self.err, stream, self.step_options, k_new.stride(0),
                                   q.stride(0), self.bt.stride(0))

    def _rows_layers(self, q, k_new, v_new, pos_dev, seq_lens_dev, out, stream, rows, ws, layer_hook=None) -> None:
        """Every layer for batch rows ``rows`` on ``stream``: one fused launch per layer, or
        (separate path) pkv_append_rope then pkv_decode_attention.  ``layer_hook(layer, phase)``
        is called around each attention launch."""
        if self.fused and layer_hook is None:
            self.fused_layers(q, k_new, v_new, seq_lens_dev, out, stream, rows, ws)
            return
        for layer in range(self.layers):
            if not self.fused:
                self.append(layer, k_new[layer], v_new[layer], q[layer], pos_dev, stream, rows)
            if layer_hook:
                layer_hook(layer, "before")
            if self.fused:
                self.fused_layer(layer, q[layer], k_new[layer], v_new[layer], seq_lens_dev, out[layer], stream,
                                 rows, ws)
            else:
                self.attention(layer, q[layer], seq_lens_dev, out[layer], stream, rows=rows, workspace=ws)
            if layer_hook:
                layer_hook(layer, "after")

    def _step_chains(self, q, k_new, v_new, pos_dev, seq_lens_dev, out, stream=None, layer_hook=None) -> None:
        """The step as micro-batch chains.  Each chain waits for the caller's stream, runs
        its layers on its own stream, and the caller's stream waits for every chain.  With
        a ``layer_hook`` the chains run one after another on the caller's stream instead, so
        that the hook's events bracket one launch each."""
        groups = list(zip(self.chain_bounds[:-1], self.chain_bounds[1:]))
        if layer_hook is not None:
            for k, rows in enumerate(groups):
                self._rows_layers(q, k_new, v_new, pos_dev, seq_lens_dev, out, stream, rows, self.chain_ws[k],
                                  layer_hook)
            return
        cur = torch.cuda.current_stream(self.device) if stream is None else stream
        fork = torch.cuda.Event()
        fork.record(cur)
        joins = []
        for k, rows in enumerate(groups):
            s = self.chain_streams[k]
            s.wait_event(fork)
            self._rows_layers(q, k_new, v_new, pos_dev, seq_lens_dev, out, s, rows, self.chain_ws[k])
            done = torch.cuda.Event()
            done.record(s)
            joins.append(done)
        for done in joins:
            cur.wait_event(done)

    def step(self, q, k_new, v_new, pos_dev, seq_lens_dev, out, stream=None, layer_hook=None) -> None:
        """One decode step over all layers.

        q: [layers][B][32][64] bf16 (rotated in place), k_new, v_new: [layers][B][8][64] bf16,
        pos_dev, seq_lens_dev: [B] int32, out: [layers][B][32][64] bf16.  The fused path
        (default) appends at seq_lens - 1 and ignores pos_dev; the separate path launches
        pkv_append_rope at pos_dev then pkv_decode_attention.  ``stream`` is a
        torch.cuda.Stream or None (the current stream).
        ``layer_hook(layer, phase)`` (optional) is called around each attention launch.
        """
        if self.chains > 1:
            self._step_chains(q, k_new, v_new, pos_dev, seq_lens_dev, out, stream, layer_hook)
            return
        self._rows_layers(q, k_new, v_new, pos_dev, seq_lens_dev, out, stream, None, self.step_ws, layer_hook)

    def steps(self, step_args, stream=None) -> None:
        """Several decode steps, ``step_args`` a sequence of (q, k_new, v_new, pos_dev,
        seq_lens_dev, out) tuples as for ``step``, in step order.  With micro-batch chains
        each chain runs its rows through every step on its own stream (forked from the
        caller's stream once, joined back once at the end); one chain runs the steps in
        order on the caller's stream.  The results equal those of ``step`` called for each
        tuple in turn."""
        step_args = list(step_args)
        if self.chains == 1:
            for args in step_args:
                self.step(*args, stream=stream)
            return
        cur = torch.cuda.current_stream(self.device) if stream is None else stream
        fork = torch.cuda.Event()
        fork.record(cur)
        joins = []
        for k, rows in enumerate(zip(self.chain_bounds[:-1], self.chain_bounds[1:])):
            s = self.chain_streams[k]
            s.wait_event(fork)
            for q, k_new, v_new, pos_dev, seq_lens_dev, out in step_args:
                self._rows_layers(q, k_new, v_new, pos_dev, seq_lens_dev, out, s, rows, self.chain_ws[k])
            done = torch.cuda.Event()
            done.record(s)
            joins.append(done)
        for done in joins:
            cur.wait_event(done)

    def run_host(self, io: "PackedIO", out_dev, out_host, stream=None) -> None:
        """End-to-end step: one copy of the step's inputs (q, k_new, v_new, pos, seq_lens, packed
        back to back in pinned host memory) to the device, the step, one copy of the output back
        to pinned host memory; all on the kernels' stream."""
        io.dev.copy_(io.host, non_blocking=True)
        d = io.d
        self.step(d["q"], d["k_new"], d["v_new"], d["pos"], d["seq_lens"], out_dev, stream)
        out_host.copy_(out_dev, non_blocking=True)

    def step_graphs(self, io: "PackedIO", out_devs, group: int = 1, pipelined: bool = False) -> list:
        """Captured CUDA graphs for ``run_host_steps``: with K = len(out_devs) buffers (a
        multiple of ``group``), graph j runs ``group`` consecutive steps, the i-th on device
        input buffer j * group + i of ``io`` into ``out_devs[j * group + i]`` (``pipelined``:
        through ``steps``, the chains joined once per graph).  Capture after a first eager
        pass (kernel attributes and tensor maps are set up outside any capture)."""
        K = len(out_devs)
        if group < 1 or K % group:
            raise ValueError(f"{K} buffers do not split into graphs of {group} steps")
        graphs = []
        for j in range(K // group):
            args = []
            for k in range(j * group, (j + 1) * group):
                d = io.buffer(k)
                args.append((d["q"], d["k_new"], d["v_new"], d["pos"], d["seq_lens"], out_devs[k]))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                if pipelined:
                    self.steps(args)
                else:
                    for a in args:
                        self.step(*a)
            graphs.append(g)
        return graphs

    def run_host_steps(self, io: "PackedIO", out_devs, out_host, steps: int, stream=None, graphs=None,
                       group: int = 1) -> None:
        """``steps`` end-to-end steps, each with its own copy of the inputs from pinned host
        memory and its own copy of the output back, through K = len(out_devs) rotating
        buffers: step s reads device input buffer s % K (``io.buffer(s % K)``) and writes
        ``out_devs[s % K]``.  Host-to-device copies run on one copy stream and device-to-host
        copies on another, so that the inputs of the next steps arrive and earlier outputs
        leave while step s computes.  A buffer is refilled only after the step that used it
        has finished, and an output buffer is rewritten only after its copy to the host has
        finished.  ``out_host`` receives the outputs in step order and ends holding the last
        step's.
        With ``graphs`` (from ``step_graphs(io, out_devs, group)``) the steps' kernels replay
        those graphs, ``group`` steps per replay, and the copies stay plain stream operations
        between the replays: inside a captured graph, copy nodes delay the kernels beside them
        (measured on GB300: about 10 us per node plus part of the copy), while stream copies
        overlap them; more steps per replay means fewer graph boundaries (each costs a few
        microseconds of idle GPU).  ``steps`` must then be a multiple of ``group``, and K of
        2 x ``group`` lets one group's copies overlap the other group's compute."""
        cur = torch.cuda.current_stream(self.device) if stream is None else stream
        if not hasattr(self, "_h2d"):
            self._h2d, self._d2h = torch.cuda.Stream(device=self.device), torch.cuda.Stream(device=self.device)
        K = len(out_devs)
        if K < 2:
            raise ValueError("run_host_steps needs at least two output buffers")
        if graphs is not None and (len(graphs) * group != K or steps % group):
            raise ValueError("graphs, group, buffers and steps do not match")
        devs = [io.buffer(k) for k in range(K)]
        raws = [io.raw(k) for k in range(K)]
        start = torch.cuda.Event()
        start.record(cur)
        self._h2d.wait_event(start)
        self._d2h.wait_event(start)
        ready = [torch.cuda.Event() for _ in range(steps)]
        done = [torch.cuda.Event() for _ in range(steps)]
        sent = [torch.cuda.Event() for _ in range(steps)]
        lead = K - 1 if graphs is None else K - group   # uploads issued ahead of the step in progress

        def upload(s):
            if s >= K:
                self._h2d.wait_event(done[s - K])      # the step that last read this buffer
            with torch.cuda.stream(self._h2d):
                raws[s % K].copy_(io.host, non_blocking=True)
            ready[s].record(self._h2d)

        issued = 0
        for s in range(steps):
            first = graphs is None or s % group == 0
            while first and issued < min(steps, s + lead + (1 if graphs is None else group)):
                upload(issued)
                issued += 1
            if graphs is None:
                cur.wait_event(ready[s])
                if s >= K:
                    cur.wait_event(sent[s - K])        # this output buffer has left for the host
                d = devs[s % K]
                self.step(d["q"], d["k_new"], d["v_new"], d["pos"], d["seq_lens"], out_devs[s % K], cur)
                done[s].record(cur)
            elif first:
                # the copy streams run their copies in order: the group's last upload and the
                # send out of the last buffer it reuses imply all the others
                last = s + group - 1
                cur.wait_event(ready[last])
                if last >= K:
                    cur.wait_event(sent[last - K])
                with torch.cuda.stream(cur):
                    graphs[(s % K) // group].replay()
                done[s].record(cur)
                for t in range(s + 1, s + group):
                    done[t] = done[s]
            self._d2h.wait_event(done[s])
            with torch.cuda.stream(self._d2h):
                out_host.copy_(out_devs[s % K], non_blocking=True)
            sent[s].record(self._d2h)
        cur.wait_event(sent[steps - 1])
        cur.wait_event(ready[steps - 1])

    def check_errors(self):
        return pkv.pkv_check_device_error(self.err)


def chain_bounds(batch: int, chains: int, seq_lens=None) -> list:
    """Row bounds [0 = r_0 < r_1 < ... < r_K = batch] of K contiguous micro-batch chains.
    Without lengths the rows are split evenly; with them, r_k is the cut whose running page
    count is nearest to k/K of the total (every chain keeps at least one row)."""
    if not 1 <= chains <= batch:
        raise ValueError(f"chains must be in [1, batch], not {chains}")
    if seq_lens is None or chains == 1:
        return [int(x) for x in np.linspace(0, batch, chains + 1).round().astype(int)]
    pages = (np.asarray(seq_lens, dtype=np.int64).clip(min=0) + wl.PAGE_SIZE - 1) // wl.PAGE_SIZE
    cum = np.cumsum(pages)
    total = int(cum[-1]) if batch else 0
    bounds = [0]
    for k in range(1, chains):
        target = total * k / chains
        i = int(np.searchsorted(cum, target, side="left"))  # first row whose running count reaches it
        r = i + 1 if i == 0 or abs(cum[min(i, batch - 1)] - target) <= abs(cum[i - 1] - target) else i
        r = max(r, bounds[-1] + 1)          # at least one row per chain
        r = min(r, batch - (chains - k))    # leave a row for every later chain
        bounds.append(r)
    bounds.append(batch)
    return bounds


class PackedIO:
    """A step's inputs packed back to back (256-byte aligned) in one pinned host buffer and
    device buffers of the same layout, so that the end-to-end step moves them with one copy.
    ``h[name]`` / ``d[name]`` are host / device views with the tensors' shapes and dtypes;
    ``buffer(k)`` / ``raw(k)`` are the views / bytes of device buffer k (allocated on first
    use; buffer 0 is ``d``)."""

    def __init__(self, tensors: dict, device):
        offsets, off = {}, 0
        for name, t in tensors.items():
            offsets[name] = off
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=device)
        self.bytes = sum(t.numel() * t.element_size() for t in tensors.values())
        self._layout = {name: (offsets[name], t.numel() * t.element_size(), t.dtype, t.shape)
                        for name, t in tensors.items()}
        self.h = {}
        for name, (o, n, dtype, shape) in self._layout.items():
            self.h[name] = self.host[o:o + n].view(dtype).view(shape)
            self.h[name].copy_(tensors[name].cpu())
        self._raws = [self.dev]
        self._views = [self._viewsof(self.dev)]
        self.d = self._views[0]

    def _viewsof(self, raw) -> dict:
        return {name: raw[o:o + n].view(dtype).view(shape) for name, (o, n, dtype, shape) in self._layout.items()}

    def raw(self, k: int):
        while len(self._raws) <= k:
            self._raws.append(torch.empty_like(self.dev))
            self._views.append(self._viewsof(self._raws[-1]))
        return self._raws[k]

    def buffer(self, k: int) -> dict:
        self.raw(k)
        return self._views[k]

    def second(self) -> dict:
        """Views of device buffer 1."""
        return self.buffer(1)
