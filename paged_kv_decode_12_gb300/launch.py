"""Launch configuration of the fused decode step per workload and KV page format.

These are the settings the benchmark times and the full-size parity tests run:
pages per work unit, TMA ring depth per warp, largest-first unit dispatch and the
number of micro-batch chains.  Each was chosen by measurement on GB300. The fixed
chunking keeps results batch invariant, because it depends only on each sequence's
own length. None of the settings changes a result bit.
"""
from __future__ import annotations

# pages per work unit (swept over 8..128 per workload; b64 together with its chains:
# with 8 chains a launch holds 8 sequences, and 20-page units shorten each unit's
# serial chain of page round trips)
CHUNK = {"tiny": 1, "b256": 128, "b64": 20, "b8": 16, "trace": 32}
# TMA stages per warp on the grid schedule, BF16 pages (4 KiB each)
RING = {"tiny": 2, "b256": 3, "b64": 2, "b8": 2, "trace": 2}
# TMA stages per warp, FP8 pages (units of 2176 B); b256 with 2 chains: ring 2 / 3 / 4 give
# 1.352 / 1.337 / 1.320 ms per step (3 or 4 chains: the same)
RING_FP8 = {"tiny": 2, "b256": 4, "b64": 2, "b8": 2, "trace": 2}
# largest-first unit dispatch (PKV_STEP_SORTED): a gain on a ragged one-wave layer run as
# one launch (b8); with micro-batch chains the grid order is faster (b64), and on b256
# every unit has the same size
SORTED = {"tiny": True, "b256": False, "b64": False, "b8": True, "trace": False}
# micro-batch chains: independent per-layer launch chains over contiguous row groups,
# each on its own stream, so that one group's layer tail overlaps another's streaming.
# Every chain adds a launch per layer: past 8 chains b64 gains nothing in multi-step
# graphs and loses at one step per graph.  The trace launches eagerly from the host each
# step (one library call per chain for all layers): 2 chains give +5 % device time and
# +3 % wall time on the continuous BF16 trace (+18 % / +15 % static), 4 chains lose; FP8
# pages gain 3 % of device time and lose 1 % of wall time, so they keep one
CHAINS = {"tiny": 2, "b256": 2, "b64": 8, "b8": 1, "trace": 2}
CHAINS_FP8 = {"tiny": 2, "b256": 2, "b64": 8, "b8": 1, "trace": 1}
# the two named calls per layer (pkv_append_rope, then pkv_decode_attention): twice the
# launches, whose latencies more chains hide (b64: 16 chains 0.205 ms per step, 8 chains 0.215)
CHAINS_SEPARATE = {"tiny": 2, "b256": 2, "b64": 16, "b8": 1, "trace": 1}


def chains(name: str, kv: str = "bf16", path: str = "fused") -> int:
    """Micro-batch chains of workload ``name`` for ``kv`` pages on the fused or separate path."""
    if path == "separate":
        return CHAINS_SEPARATE[name]
    return (CHAINS if kv == "bf16" else CHAINS_FP8)[name]


def config(name: str, kv: str = "bf16", path: str = "fused") -> dict:
    """Keyword arguments of ``harness.setup`` for workload ``name`` with ``kv`` pages."""
    if kv not in ("bf16", "fp8"):
        raise ValueError(f"kv must be 'bf16' or 'fp8', not {kv!r}")
    if path not in ("fused", "separate"):
        raise ValueError(f"path must be 'fused' or 'separate', not {path!r}")
    return {"pages_per_chunk": CHUNK[name], "ring": (RING if kv == "bf16" else RING_FP8)[name],
            "sorted_units": SORTED[name], "chains": chains(name, kv, path), "kv": kv, "fused": path == "fused"}
