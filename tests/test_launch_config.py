"""Host logic of the launch configuration: the per-workload settings and the
micro-batch chain cuts (engine.chain_bounds).  CPU only."""
import numpy as np
import pytest

from paged_kv_decode_12_gb300 import launch
from paged_kv_decode_12_gb300 import workloads as wl
from paged_kv_decode_12_gb300.engine import chain_bounds


def test_launch_config_covers_every_workload():
    for name in ("tiny", "b8", "b64", "b256", "trace"):
        for kv in ("bf16", "fp8"):
            for path in ("fused", "separate"):
                c = launch.config(name, kv, path)
                assert set(c) == {"pages_per_chunk", "ring", "sorted_units", "chains", "kv", "fused"}
                assert 1 <= c["pages_per_chunk"] <= 128 and c["ring"] in (2, 3, 4) and c["chains"] >= 1
                assert c["fused"] == (path == "fused") and c["chains"] == launch.chains(name, kv, path)
    with pytest.raises(ValueError):
        launch.config("b64", "int4")
    with pytest.raises(ValueError):
        launch.config("b64", "bf16", "split")


def test_chain_bounds_even_split():
    assert chain_bounds(64, 4) == [0, 16, 32, 48, 64]
    assert chain_bounds(5, 2) == [0, 2, 5] or chain_bounds(5, 2) == [0, 3, 5]
    assert chain_bounds(8, 1) == [0, 8] and chain_bounds(3, 3) == [0, 1, 2, 3]
    with pytest.raises(ValueError):
        chain_bounds(4, 5)
    with pytest.raises(ValueError):
        chain_bounds(4, 0)


@pytest.mark.parametrize("name", ["b8", "b64", "b256"])
@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
def test_chain_bounds_balance_pages(name, K):
    w = wl.make_workload(name)
    b = chain_bounds(w.batch, K, w.seq_lens)
    assert b[0] == 0 and b[-1] == w.batch and len(b) == K + 1
    assert all(x < y for x, y in zip(b[:-1], b[1:]))           # every chain keeps a row
    pages = -(-w.seq_lens.astype(np.int64) // wl.PAGE_SIZE)
    cum = np.concatenate([[0], np.cumsum(pages)])
    biggest = int(pages.max())
    if K == w.batch:                                            # one row per chain: nothing to balance
        return
    for k in range(1, K):                                       # each cut within one row of k/K
        assert abs(cum[b[k]] - cum[-1] * k / K) <= biggest


def test_chain_bounds_degenerate_lengths():
    assert chain_bounds(5, 2, [0, 0, 0, 0, 0]) == [0, 1, 5]
    assert chain_bounds(4, 4, [2048, 1, 1, 1]) == [0, 1, 2, 3, 4]
    assert chain_bounds(3, 2, [1, 1, 4000]) == [0, 2, 3]
    assert chain_bounds(3, 2, [-5, 16, 16]) in ([0, 1, 3], [0, 2, 3])
