"""bench.py's command-line overrides, on the CPU: the workload a line
measures is the one its JSON names."""
import argparse
import json
import os
import subprocess
import sys

import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ns(**kw):
    base = dict(num_seqs=0, num_blocks=0, block_size=0, dtype="bf16", head_dim=0, workload="mha",
                prefix_len=0, num_shared=0)
    base.update(kw)
    return argparse.Namespace(**base)


def test_overrides_reach_the_workload_and_the_json_line():
    ns = _ns(dtype="f32", head_dim=96, num_seqs=4, workload="gqa")
    ov = bench.overrides(ns)
    assert ov["dtype"] == torch.float32 and ov["head_dim"] == 96
    assert ov["num_seqs"] == 4 and ov["num_shared"] == 1          # gqa keeps a shared prefix
    assert json.loads(json.dumps(bench.overrides_json(ns))) == {
        "num_seqs": 4, "num_shared": 1, "dtype": "f32", "head_dim": 96}
    assert bench.overrides(_ns()) == {}
    # the shared-prefix size of the gqa batch
    ov = bench.overrides(_ns(workload="gqa", prefix_len=4096, num_shared=64))
    assert ov == {"prefix_len": 4096, "num_shared": 64}
    from paged_kv_cache_109_gb300 import workloads
    wl = workloads.make("gqa", num_seqs=16, num_blocks=8192, **ov | {"num_shared": 8})
    assert wl.prefix_groups[0][1] == 4096 // wl.block_size


def test_block_size_sweep_keeps_pool_bytes():
    for w, (nb, bs) in {"mha": (8192, 16), "long": (16384, 32)}.items():
        ov = bench.overrides(_ns(workload=w, block_size=64))
        assert ov["block_size"] * ov["num_blocks"] == nb * bs


def test_decode_only_flags_are_refused_elsewhere():
    for w in ("copy", "prefill"):
        r = subprocess.run([sys.executable, "bench.py", "--workload", w, "--dtype", "f32"],
                           capture_output=True, text=True, cwd=ROOT)
        assert r.returncode != 0 and "decode workloads" in r.stderr


def test_default_line_is_the_long_context_decode():
    """With no flags the bench measures the long-context GQA batch (the
    largest single-GPU workload, 2 GiB of K/V per decode)."""
    args = bench.make_parser().parse_args([])
    assert args.workload == "long" and args.gpus == 1 and args.warmup >= 3
    assert "131072" in bench.WORKLOAD_TEXT[args.workload]
    # the roofline block is long enough to be a per-call mean, not a sample
    assert bench.ROOF_MIN_CALLS >= 200 and bench.ROOF_SAMPLED >= 20


def test_reference_arm_describes_the_same_workload():
    """The reference arm's config is built by the GPU arm's own function, so
    the two lines of one command name the same workload."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "mha",
                        "--num-seqs", "2", "--num-blocks", "512", "--steps", "1",
                        "--cpu-seconds", "0.2"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    from paged_kv_cache_109_gb300 import workloads
    args = bench.make_parser().parse_args(["--workload", "mha", "--num-seqs", "2",
                                           "--num-blocks", "512"])
    wl = workloads.make("mha", **bench.overrides(args))
    assert line["config"] == json.loads(json.dumps(bench.decode_config(args, wl, 1)))
    assert line["impl"] == "reference" and line["config"]["num_seqs"] == 2


def test_decode_steps_write_inside_the_decode_call():
    """The decode workloads' steps add one token per sequence at its last
    position, so by default their write goes inside the decode call
    (pa_decode_append); continuous batching, whose steps also write a chunk,
    keeps the cache-write call."""
    import pytest
    from paged_kv_cache_109_gb300 import workloads
    small = {"mha": dict(num_seqs=3, num_blocks=512),
             "gqa": dict(num_seqs=8, num_shared=2, num_blocks=4096),
             "long": dict(num_seqs=1, seq_len=2000),
             "cb": dict(num_seqs=4, max_len0=100, chunk=30, num_steps=2, num_blocks=256)}
    for name, kw in small.items():
        wl = workloads.make(name, **kw)
        args = bench.make_parser().parse_args(["--workload", name])
        want = "slot_mapping" if name == "cb" else "append"
        assert bench.appends_only(wl) == (name != "cb")
        assert bench.write_mode(args, wl) == want
        assert bench.write_mode(bench.make_parser().parse_args(
            ["--workload", name, "--positions"]), wl) == "positions"
        assert bench.write_mode(bench.make_parser().parse_args(
            ["--workload", name, "--write", "slot_mapping"]), wl) == "slot_mapping"
    with pytest.raises(SystemExit):
        bench.write_mode(bench.make_parser().parse_args(["--workload", "cb", "--write",
                                                         "append"]), wl)
