"""bench.py's argument resolution (CPU only): the per-workload launch settings it
fills in are the ones in paged_kv_decode_12_gb300/launch.py, explicit flags win, and
combinations the path does not run are refused before any GPU work."""
import pytest

import bench
from paged_kv_decode_12_gb300 import launch


@pytest.fixture
def captured(monkeypatch):
    seen = {}

    def grab(name):
        def run(args):
            seen["arm"], seen["args"] = name, args
            return 0
        return run

    monkeypatch.setattr(bench, "run_pkv", grab("pkv"))
    monkeypatch.setattr(bench, "run_trace", grab("trace"))
    monkeypatch.setattr(bench, "run_reference", grab("reference"))
    return seen


@pytest.mark.parametrize("config", ["b256", "b64", "b8"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_defaults_follow_launch_table(captured, config, kv):
    assert bench.main(["--config", config, "--kv", kv]) == 0
    a, want = captured["args"], launch.config(config, kv)
    assert captured["arm"] == "pkv"
    assert (a.pages_per_chunk, a.ring, a.sorted, a.chains) == \
        (want["pages_per_chunk"], want["ring"], want["sorted_units"], want["chains"])


def test_explicit_flags_win(captured):
    bench.main(["--chains", "1", "--ring", "4", "--pages-per-chunk", "64", "--unsorted"])
    a = captured["args"]
    assert (a.chains, a.ring, a.pages_per_chunk, a.sorted) == (1, 4, 64, False)
    bench.main(["--config", "b64", "--sorted"])
    assert captured["args"].sorted is True


def test_separate_path_options(captured):
    # the separate path (pkv_append_rope + pkv_decode_attention) takes the workload's chains
    bench.main(["--path", "separate", "--config", "b64"])
    assert captured["args"].chains == launch.CHAINS_SEPARATE["b64"] and not captured["args"].split_merge
    bench.main(["--path", "separate", "--chains", "2", "--split-merge"])
    a = captured["args"]
    assert a.chains == 2 and a.split_merge and a.sorted is False
    with pytest.raises(SystemExit):     # the two-kernel form belongs to the separate path
        bench.main(["--split-merge"])
    with pytest.raises(SystemExit):
        bench.main(["--sorted", "--unsorted"])


def test_trace_and_reference_arms(captured):
    bench.main(["--config", "trace"])
    assert captured["arm"] == "trace" and captured["args"].chains == launch.CHAINS["trace"]
    bench.main(["--impl", "reference", "--config", "b64"])
    assert captured["arm"] == "reference" and captured["args"].chains == launch.CHAINS["b64"]


def test_extra_specs_and_pipelined_settings(captured):
    assert bench.parse_extra("b64") == ("b64", "bf16", "fused", False, False)
    assert bench.parse_extra("b64:fp8:pipelined") == ("b64", "fp8", "fused", False, True)
    assert bench.parse_extra("b64:split-merge") == ("b64", "bf16", "separate", True, False)
    for bad in ("b64:nope", "trace", "b99"):
        with pytest.raises(SystemExit):
            bench.parse_extra(bad)
    for spec in bench.EXTRA_DEFAULT:     # every default extra parses
        bench.parse_extra(spec)
    bench.main(["--config", "b64", "--pipelined"])
    args = captured["args"]
    assert args.pipelined is True
    a = bench.run_settings(args, "b64", pipelined=False)
    assert a.pipelined is False and a.chains == launch.CHAINS["b64"] and args.pipelined is True
