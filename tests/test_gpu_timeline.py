"""The per-CTA timeline build (include/pkv_timeline.h) records one consistent entry
per work unit of a fused-step launch: monotone stamps, the unit's page count, and
nothing for CTAs without a unit.  The default library does not export it."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_timeline_records_every_unit_once():
    import subprocess
    import sys

    # a fresh process, so that the timeline library is the only libpkv it loads
    code = r"""
import numpy as np, torch
from paged_kv_decode_12_gb300 import _build, pkv
pkv.LIB_PATH = _build.build(timeline=True)
from paged_kv_decode_12_gb300 import harness, timeline
dw = harness.setup("tiny", pages_per_chunk=1, ring=2)
dw.step(); torch.cuda.synchronize()
n = 8 * dw.w.batch * dw.w.max_blocks
stamps, meta = timeline._read(n)
live = meta[:, 0] >= 0
expect = 8 * sum(-(-int(L) // 16) for L in dw.w.seq_lens)   # one unit per (page, head) at 1 page a chunk
assert live.sum() == expect, (live.sum(), expect)
t = stamps[live].astype(np.int64)
assert np.all(np.diff(t, axis=1) >= 0) and np.all(t[:, 0] > 0)
assert np.all(meta[live, 3] == 1) and np.all(meta[live, 0] < torch.cuda.get_device_properties(0).multi_processor_count)
print(timeline.summarize(stamps, meta, torch.cuda.get_device_properties(0).multi_processor_count))
"""
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


def test_default_library_has_no_timeline():
    from paged_kv_decode_12_gb300 import _build, pkv

    _build.build()
    lib = ctypes.CDLL(pkv.LIB_PATH)
    assert not hasattr(lib, "pkv_timeline_read")
