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
    base = dict(num_seqs=0, num_blocks=0, block_size=0, dtype="bf16", head_dim=0, workload="mha")
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
