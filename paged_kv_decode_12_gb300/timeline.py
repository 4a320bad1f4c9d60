"""Per-CTA timeline of one layer of the fused decode step (grid schedule).

    python -m paged_kv_decode_12_gb300.timeline --config b64 [--pages-per-chunk 32]
           [--ring 2] [--sorted] [--save timeline.npz]

Builds libpkv_timeline.so (the library compiled with -DPKV_TIMELINE, see
include/pkv_timeline.h), runs two decode steps of the named workload as a CUDA
graph, reads the records of the last launch (the last layer) and prints where its
time goes: when CTAs entered relative to the release of the previous launch, the
page-loop and finish times by unit size, the SMs' loads and end times, the number
of CTAs streaming over time.  A measurement aid only; the default library has no
timeline code.
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np


def _read(n: int):
    from . import pkv

    L = pkv.lib()
    L.pkv_timeline_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.pkv_timeline_read.restype = ctypes.c_int
    stamps = np.zeros((n, 5), dtype=np.uint64)
    meta = np.zeros((n, 4), dtype=np.int32)
    got = L.pkv_timeline_read(stamps.ctypes.data, meta.ctypes.data, n)
    if got != n:
        raise RuntimeError(f"pkv_timeline_read returned {got}")
    return stamps, meta


def summarize(stamps: np.ndarray, meta: np.ndarray, num_sms: int) -> str:
    """Text summary of one launch's records (CTAs with SM -1 are skipped)."""
    live = meta[:, 0] >= 0
    t = stamps[live].astype(np.int64)
    m = meta[live]
    base = t[:, 2].min()                       # first CTA released from the dependency wait
    rel = (t - base) / 1000.0                  # microseconds
    pages = m[:, 3]
    loop = rel[:, 3] - rel[:, 2]
    finish = rel[:, 4] - rel[:, 3]
    out = [f"units {int(live.sum())} of {len(meta)} CTAs; times in us from the first release"]
    for name, col in (("entry", 0), ("unit known", 1), ("released", 2), ("pages done", 3), ("end", 4)):
        out.append(f"  {name:10s} min {rel[:, col].min():7.2f}  p50 {np.median(rel[:, col]):7.2f}  "
                   f"max {rel[:, col].max():7.2f}")
    edges = [1, 2, 5, 10, 20, 33, 65, 129]
    for lo, hi in zip(edges[:-1], edges[1:]):
        sel = (pages >= lo) & (pages < hi)
        if sel.any():
            out.append(f"  pages [{lo:3d},{hi:3d}): {int(sel.sum()):5d} units, loop p50 {np.median(loop[sel]):6.2f} "
                       f"max {loop[sel].max():6.2f}, finish p50 {np.median(finish[sel]):5.2f} "
                       f"max {finish[sel].max():5.2f}, end max {rel[sel, 4].max():6.2f}")
    sm = m[:, 0]
    ends = np.array([rel[sm == s, 4].max() if (sm == s).any() else 0.0 for s in range(num_sms)])
    load = np.array([pages[sm == s].sum() for s in range(num_sms)])
    units = np.array([(sm == s).sum() for s in range(num_sms)])
    out.append(f"  per SM: end p50 {np.median(ends):.2f} max {ends.max():.2f}; pages min {load.min()} "
               f"p50 {int(np.median(load))} max {load.max()}; units min {units.min()} max {units.max()}")
    grid = np.arange(0.0, rel[:, 4].max() + 1.0, 1.0)
    streaming = [int(((rel[:, 2] <= x) & (rel[:, 3] > x)).sum()) for x in grid]
    out.append("  CTAs in their page loop, per us: " + " ".join(str(v) for v in streaming))
    return "\n".join(out)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--config", default="b64", choices=["tiny", "b8", "b64", "b256"])
    ap.add_argument("--pages-per-chunk", type=int, default=32)
    ap.add_argument("--ring", type=int, default=2, choices=[0, 2, 3, 4])
    ap.add_argument("--sorted", action="store_true")
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--save", default=None, help="write the raw records to this .npz file")
    args = ap.parse_args(argv)

    from . import _build, pkv

    pkv.LIB_PATH = _build.build(timeline=True)
    import torch

    from . import harness

    dw = harness.setup(args.config, pages_per_chunk=args.pages_per_chunk, ring=args.ring, layers=args.layers,
                       sorted_units=args.sorted)
    harness.warm(dw, 2)
    dw.reset_q()
    cap = harness.capture_steps(dw, 2)
    cap.graph.replay()
    torch.cuda.synchronize()
    st, flag = dw.eng.check_errors()
    if st != pkv.PKV_OK:
        raise SystemExit(f"device error flag {flag:#x}")
    n = 8 * dw.w.batch * ((dw.w.max_blocks + args.pages_per_chunk - 1) // args.pages_per_chunk)
    if n > 16384:
        raise SystemExit(f"{n} CTAs: more than the 16384 records of the timeline")
    stamps, meta = _read(n)
    if args.save:
        np.savez(args.save, stamps=stamps, meta=meta)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    print(f"{args.config}: pages_per_chunk {args.pages_per_chunk}, ring {args.ring}, sorted {args.sorted}, "
          f"last layer of a {dw.w.layers}-layer step")
    print(summarize(stamps, meta, sms))
    dw.eng.close()
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
