#!/usr/bin/env python
"""Benchmark: one step = pa_write_kv of the step's new tokens + pa_decode of
the whole batch (every row of the hot path), on synthetic inputs resident in
HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long|mha|gqa|cb|...]
                    [--impl ours|reference] [--partition P]

The default workload is the long-context GQA batch (4 x 131072 tokens, the
largest single-GPU case, 2 GiB of K/V per decode).

Metric: paged-decode KV GB/s = algorithmic bytes of the step / step time;
also % of the measured HBM peak and decode tokens/s per layer (sequences
decoded per second).  For N > 1 (torchrun) every rank runs its own replica
of the batch (the path shards by sequence with no exchange): value is the
sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_109_gb300 import workloads  # noqa: E402

METRIC = "paged decode KV GB/s and % of GB300 HBM peak; decode tokens/s per layer"
L2_BYTES = 129 * 1024 * 1024
ROOF_MIN_CALLS = 200    # the roofline block: at least this many back-to-back decode calls
ROOF_MIN_MS = 250.0     # ... and at least this long (several clock samples)
ROOF_SAMPLED = 50       # isolated decode calls, each between its own events (quantiles)
ROOF_STEP_SLACK = 1.02  # self-check: per-call time <= ms_per_step x this
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0     # GB300 HBM3e nominal, reported beside the measured denominator
F32_BOUND = 1e-5             # fp32 outputs: max abs error against the fp64 oracle
WORKLOAD_TEXT = {
    "mha": "MHA decode bf16: 32 seqs, Hq=Hkv=32, D=128, B=16, T~U[128,2048], 8192-block "
           "shuffled pool; step = write 1 new token per seq + decode",
    "gqa": "GQA decode bf16: 128 seqs, Hq=32, Hkv=8, D=128, B=16, T~lognormal(median 1024, "
           "sigma 1) cap 8192, 32 seqs share a 512-token prefix; 65536-block pool; "
           "step = write 1 new token per seq + decode",
    "long": "long-context GQA decode bf16: 4 seqs x 131072, Hq=64, Hkv=8, D=128, B=32, "
            "16384-block pool; step = write 1 new token per seq + split-K decode + merge",
    "cb": "continuous batching bf16: 256 seqs, Hq=32, Hkv=8, D=128, B=16, T0~U[1,4096]; "
          "step = write 2304 tokens (1 per seq + 2048-token chunk) + decode all 256; "
          "10 distinct steps cycled",
    "prefill": "chunked prefill bf16: 8 seqs with history T0~U[1,4096] each taking a "
               "2048-token chunk, Hq=32, Hkv=8, D=128, B=16; step = write the 16384 chunk "
               "tokens + causal multi-query attention from every chunk token",
    "copy": "block copy inside one pool (copy-on-write), bf16: 8192 disjoint (src, dst) pairs "
            "of B=16, Hkv=8, D=128 blocks (64 KiB of K+V each) in a 65536-block pool; "
            "step = one pa_copy_blocks call",
    "swap": "swap through page-locked host memory, bf16: 2048 blocks of B=16, Hkv=8, D=128 "
            "out to a host pool and 2048 back; step = two pa_copy_blocks calls",
}


# ---- byte model ---------------------------------------------------------------

def step_bytes(wl, k: int, split_traffic: bool = True, shared_prefix: bool = False,
               partition: int = 0, fused: bool = False) -> dict:
    """Algorithmic bytes of step k (see the design notes for the model).
    With ``split_traffic`` the split-K partial write + read at ``partition``
    tokens (0: the library's automatic size, asked of libpa.so) is included;
    with ``shared_prefix`` the partials of the shared-prefix decode (every
    group member writes its group's prefix partitions and its own).  With
    ``fused`` the write is pa_decode_append's, which reads no slot mapping."""
    st = wl.steps[k]
    e = wl.elem_bytes
    row = wl.head_dim * e
    per_tok = 2 * wl.num_kv_heads * row                 # K + V of one token, one layer
    lens = st.seq_lens.to(torch.int64)
    logical_kv = int(lens.sum()) * per_tok
    # unique: each physical block's valid rows counted once (shared prefix)
    bs = wl.block_size
    seen = {}
    for i, t in enumerate(lens.tolist()):
        for lb in range(-(-t // bs)):
            b = int(st.block_tables[i, lb])
            seen[b] = max(seen.get(b, 0), min(bs, t - lb * bs))
    unique_kv = sum(seen.values()) * per_tok
    n, hq = st.q.shape[0], wl.num_q_heads
    q_out = 2 * n * hq * row
    tables = sum(-(-t // bs) for t in lens.tolist()) * 4 + n * 4
    split, ws, part = 0, 0, None
    if split_traffic:
        import paged_kv_cache_109_gb300 as pa
        ws = pa.decode_workspace_bytes(n, hq, int(lens.max()), wl.k_cache, partition)
        part = partition or pa.decode_partition_tokens(n, hq, int(lens.max()), wl.k_cache)
        member_pk = {}
        if shared_prefix:
            for members, blocks in wl.prefix_groups:
                for i in members:
                    member_pk[i] = blocks * bs
        # each split sequence writes and re-reads (D + 2) floats per partition and head
        for i, t in enumerate(lens.tolist()):
            if i in member_pk:
                pk = member_pk[i]
                parts = -(-pk // part) + -(-max(0, t - pk) // part)
                split += 2 * parts * hq * (wl.head_dim + 2) * 4
                continue
            parts = -(-t // part)
            if parts > 1:
                split += 2 * parts * hq * (wl.head_dim + 2) * 4
    n_tok = st.slot_mapping.numel()
    # read k,v + write cache rows (+ the slot, unless the decode call appends)
    write = n_tok * (2 * per_tok + (0 if fused else 8))
    return {"logical_kv": logical_kv, "unique_kv": unique_kv, "decode": unique_kv + q_out +
            tables + split, "decode_logical": logical_kv + q_out + tables + split,
            "write": write, "workspace": ws, "partition": part}


# ---- clocks --------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max((num(r[3]) or 0) for r in rows)}


# sources of the kernels whose traffic is recorded for the decode lines (the
# TMA kernel and the merge, with the sizing in decode_config.cuh; the tiled
# kernel never runs on those bf16 D=128 workloads)
KERNEL_SOURCES = ("decode_tma_mma.cuh", "ptx.cuh", "merge.cuh", "decode_generic.cuh",
                  "common.cuh", "decode_config.cuh")


# sources of the kernels whose traffic is recorded for the prefill and copy lines
PREFILL_SOURCES = ("prefill_ws.cuh", "prefill_args.cuh", "ptx.cuh", "common.cuh",
                   "decode_generic.cuh")
COPY_SOURCES = ("write_kv.cuh", "common.cuh", "ptx.cuh")


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_109_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch of the line's dominant kernel from the committed
    ncu summary, or None when there is none for this workload or that
    kernel's sources (the record's list, else the decode kernel's) changed."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    sources = tuple(rec.get("kernel_sources", KERNEL_SOURCES))
    if rec.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return rec.get("dram_bytes_per_launch")


def measured_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---- ranks (one process per GPU; replicas) -----------------------------------

def rank_barrier() -> None:
    """All ranks meet here (no-op for a single process)."""
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks (the slowest rank's timed region); x with
    one process.  ``device`` holds the reduction buffer: the GPU under NCCL,
    the CPU under gloo."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    if torch.distributed.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---- CPU oracle (reference arm and cpu_baseline) ----------------------------------

def time_oracle(wl, budget_s: float, max_reps: int = 50, gpu_outs=None,
                one_core_s: float = 0.0) -> dict:
    """The oracle, as it stands, on the host cores: full steps (write + decode
    of every (sequence, head)) repeated until ~budget_s seconds.  With
    ``gpu_outs`` (the GPU's output of each step), each step's oracle output is
    also compared with the GPU's (outside the timed span): the largest
    absolute error and the largest ratio to the bound (bf16 3e-3 + 1e-2 |ref|,
    fp32 1e-5)."""
    import oracle
    threads = oracle.max_threads()
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    done_bytes, reps, elapsed = 0, 0, 0.0
    err_abs, err_ratio, checked = 0.0, 0.0, set()
    while reps < max_reps:
        k = reps % len(wl.steps)
        st = wl.steps[k]
        t0 = time.perf_counter()
        oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kc, vc)
        ref = oracle.decode(st.q, kc, vc, st.block_tables, st.seq_lens, wl.scale)
        elapsed += time.perf_counter() - t0
        b = step_bytes(wl, k, split_traffic=False)
        done_bytes += b["decode"] + b["write"]
        reps += 1
        if gpu_outs is not None and k not in checked:
            got = gpu_outs[k].double().cpu().numpy()
            diff = abs(got - ref)
            err_abs = max(err_abs, float(diff.max()))
            bound = F32_BOUND if wl.dtype == torch.float32 else 3e-3 + 1e-2 * abs(ref)
            err_ratio = max(err_ratio, float((diff / bound).max()))
            checked.add(k)
        if elapsed >= budget_s:
            break
    out = {"value": done_bytes / elapsed / 1e9, "unit": "GB/s", "cores": threads,
           "kind": "oracle", "seconds": round(elapsed, 3), "steps": reps,
           "sample": f"{reps} full step(s) of the {wl.name} workload (write + decode of "
                     f"all sequences and heads), fp64 C oracle with OpenMP, "
                     f"{elapsed:.1f} s"}
    # one step on one core takes about (all-core step time) x threads
    step_1core_est = elapsed / max(reps, 1) * threads
    if one_core_s > 0 and threads > 1 and step_1core_est > 2 * one_core_s:
        out["value_1_core"] = None
        out["note_1_core"] = f"skipped: one step would take about {step_1core_est:.0f} s on one core"
    elif one_core_s > 0 and threads > 1:
        # the same steps on one core, for a shorter sample
        oracle.set_threads(1)
        try:
            kc1, vc1 = wl.k_cache.clone(), wl.v_cache.clone()
            b1, r1, e1 = 0, 0, 0.0
            while r1 < max_reps and e1 < one_core_s:
                k = r1 % len(wl.steps)
                st = wl.steps[k]
                t0 = time.perf_counter()
                oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kc1, vc1)
                oracle.decode(st.q, kc1, vc1, st.block_tables, st.seq_lens, wl.scale)
                e1 += time.perf_counter() - t0
                b = step_bytes(wl, k, split_traffic=False)
                b1 += b["decode"] + b["write"]
                r1 += 1
            out["value_1_core"] = b1 / e1 / 1e9
            out["steps_1_core"] = r1
        finally:
            oracle.set_threads(threads)
    if gpu_outs is not None:
        out["max_abs_err_vs_gpu"] = err_abs
        key = "max_err_over_f32_bound" if wl.dtype == torch.float32 else "max_err_over_bf16_bound"
        out[key] = round(err_ratio, 4)
        out["steps_compared"] = len(checked)
    return out


def time_oracle_prefill(wl, budget_s: float, piece: int = 256) -> dict:
    """The oracle's chunked prefill on the host cores: the chunk write of every
    sequence, then the causal attention of the chunk rows, `piece` rows per
    call, until ~budget_s seconds (one full step is about a TFLOP in fp64).
    Rows [a, b) of sequence i's chunk are the last b - a positions of a
    sequence of length T_i - L_i + b, so each piece is a prefill call of its
    own.  value = the step's bytes as the GPU line counts them (the write,
    plus the attention's bytes scaled by the share of rows done) per second."""
    import oracle
    threads = oracle.max_threads()
    st = wl.steps[0]
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    qs, lens = st.query_start.tolist(), st.seq_lens.tolist()
    t0 = time.perf_counter()
    oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kc, vc)
    elapsed = time.perf_counter() - t0
    rows = 0
    for i in range(len(lens)):
        L = qs[i + 1] - qs[i]
        for a in range(0, L, piece):
            b = min(L, a + piece)
            t_len = lens[i] - L + b
            t0 = time.perf_counter()
            oracle.prefill(st.q[qs[i] + a:qs[i] + b], torch.tensor([0, b - a], dtype=torch.int32),
                           kc, vc, st.block_tables[i:i + 1],
                           torch.tensor([t_len], dtype=torch.int32), wl.scale)
            elapsed += time.perf_counter() - t0
            rows += b - a
            if elapsed >= budget_s:
                break
        if elapsed >= budget_s:
            break
    by = step_bytes(wl, 0, split_traffic=False)
    done = by["write"] + by["decode"] * rows / qs[-1]
    # steps: the share of one step done (the attention's rows), so that
    # seconds / steps is the time of a whole step at this rate
    return {"value": done / elapsed / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": round(elapsed, 3), "steps": round(rows / qs[-1], 4),
            "sample": f"the chunk write of all {len(lens)} sequences, then the causal prefill "
                      f"of {rows} of the {qs[-1]} chunk rows ({piece} rows per call), fp64 C "
                      f"oracle with OpenMP, {elapsed:.1f} s"}


def time_oracle_copy(args):
    """The oracle's block copy on the host, repeated for ~cpu_seconds; returns
    the timing and the workload it copied."""
    import oracle
    if args.workload == "copy":
        wl = (workloads.copy_pairs(num_blocks=args.num_blocks, num_pairs=args.num_blocks // 4)
              if args.num_blocks else workloads.copy_pairs())
    else:
        wl = workloads.copy_pairs(num_blocks=8192, num_pairs=2048)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.copy_blocks(wl.k_cache, wl.v_cache, wl.k_cache, wl.v_cache, wl.pairs)
        reps += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds or reps >= max(1, args.steps):
            break
    return {"value": reps * wl.copy_bytes() / el / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "seconds": round(el, 3), "steps": reps,
            "sample": f"{reps} oracle block-copy call(s) of {wl.pairs.shape[0]} pairs "
                      "(sequential memcpy), 1 thread"}, wl


# ---- the workload's description (shared by both arms' JSON lines) -------------------

def parallelism(world: int) -> str:
    return f"replicas x{world}" if world > 1 else "single GPU"


def appends_only(wl) -> bool:
    """Whether every step writes exactly one token per sequence, at its last
    position (a decode step): then the write can go inside the decode call."""
    for st in wl.steps:
        n = st.seq_lens.numel()
        if st.seq_ids is None or st.seq_ids.numel() != n:
            return False
        if not torch.equal(st.seq_ids, torch.arange(n, dtype=torch.int32)):
            return False
        if not torch.equal(st.positions, st.seq_lens - 1):
            return False
    return True


WRITE_TEXT = {"append": "each sequence's new token at position seq_lens - 1, written by the "
                        "decode call itself (pa_decode_append)",
              "positions": "device slots from (seq, position) (pa_write_kv_positions)",
              "slot_mapping": "slot_mapping (pa_write_kv)"}


def write_mode(args, wl) -> str:
    """How a decode step writes its new tokens: fused into the decode call
    where the steps are pure appends (automatic), else a cache-write call."""
    mode = "positions" if args.positions else args.write
    if mode == "auto":
        return "append" if appends_only(wl) else "slot_mapping"
    if mode == "append" and not appends_only(wl):
        raise SystemExit(f"--write append: the {args.workload} steps write other tokens than "
                         f"each sequence's last position")
    return mode


def decode_config(args, wl, world: int) -> dict:
    """The decode line's workload, identical in the GPU and reference arms."""
    b0 = step_bytes(wl, 0, split_traffic=False)
    return {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload,
            "overrides": overrides_json(args) or None,
            "write": WRITE_TEXT[write_mode(args, wl)],
            "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "max_seq_len": wl.max_seq_len, "seed": wl.seed,
            "block_utilization": wl.stats.get("block_utilization"),
            "shared_prefix_groups": len(wl.prefix_groups),
            "l2": f"inputs larger than L2: {b0['unique_kv'] / 2**20:.0f} MiB of K/V "
                  f"per step vs {L2_BYTES / 2**20:.0f} MiB L2",
            "parallelism": parallelism(world)}


def prefill_config(args, wl, world: int) -> dict:
    st = wl.steps[0]
    by = step_bytes(wl, 0, split_traffic=False)
    return {"workload": WORKLOAD_TEXT["prefill"], "name": "prefill",
            "overrides": overrides_json(args) or None, "num_seqs": wl.num_seqs,
            "query_rows": int(st.query_start[-1]), "max_seq_len": int(st.seq_lens.max()),
            "l2": f"inputs larger than L2: {by['unique_kv'] / 2**20:.0f} MiB of K/V",
            "parallelism": parallelism(world)}


def copy_config(args, wl, pairs_per_call: int, step_bytes_: int, world: int) -> dict:
    return {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload,
            "pairs_per_call": pairs_per_call,
            "l2": f"inputs larger than L2: {step_bytes_ / 2 / 2**20:.0f} MiB read per step",
            "parallelism": parallelism(world)}


# ---- GPU arm ------------------------------------------------------------------------

def run_ours(args, rank, world, device):
    import paged_kv_cache_109_gb300 as pa
    pa.load_library()
    wl = workloads.make(args.workload, **overrides(args))
    nsteps_wl = len(wl.steps)
    kc, vc = wl.k_cache.to(device), wl.v_cache.to(device)
    # device-resident inputs of every distinct step
    dsteps = []
    for st in wl.steps:
        dsteps.append({k: getattr(st, k).to(device) for k in
                       ("q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens",
                        "seq_ids", "positions")})
    # groups sharing leading blocks: the shared-prefix decode reads them once
    shared = bool(wl.prefix_groups) and not args.no_shared_prefix
    groups = pa.prefix_groups(wl.prefix_groups, wl.num_seqs, device) if shared else None
    # the byte model follows the path the call takes: the shared-prefix
    # partials only when the shared blocks are read once
    once = shared and pa.decode_shared_prefix_mode(wl.num_q_heads, groups.max_prefix_blocks,
                                                   kc) == 1
    mode = write_mode(args, wl)
    if mode == "append" and once:
        # the fused call runs the plain decode; where the shared-prefix decode
        # reads the shared blocks once, the step keeps it and writes first
        if args.write == "append":
            raise SystemExit("--write append: this batch's shared blocks are read once, which "
                             "the fused call does not do; use --write slot_mapping")
        mode = "slot_mapping"
    # where the shared-prefix decode would run the plain decode anyway, the
    # step's fused call is that same plain decode
    if mode == "append":
        shared = False
    part = args.partition or 0
    bytes_ = [step_bytes(wl, k, shared_prefix=once, partition=part, fused=mode == "append")
              for k in range(nsteps_wl)]
    maxlens = [int(st.seq_lens.max()) for st in wl.steps]
    ws_need = max(pa.decode_shared_prefix_workspace_bytes(wl.num_seqs, wl.num_q_heads, m,
                                                          groups.max_prefix_blocks, kc, part)
                  if shared else
                  pa.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, m, kc, part)
                  for m in maxlens)
    ws = torch.empty(max(ws_need, 256), dtype=torch.uint8, device=device)
    outs = [torch.empty_like(d["q"]) for d in dsteps]
    stream = torch.cuda.current_stream(device)

    def decode(k):
        d = dsteps[k]
        if shared:
            pa.decode_shared_prefix(d["q"], kc, vc, d["block_tables"], d["seq_lens"],
                                    maxlens[k], groups, wl.scale, out=outs[k], workspace=ws,
                                    partition_tokens=part)
        else:
            pa.decode(d["q"], kc, vc, d["block_tables"], d["seq_lens"], maxlens[k], wl.scale,
                      out=outs[k], workspace=ws, partition_tokens=part)

    def append(k):
        d = dsteps[k]
        pa.decode_append(d["q"], d["k_new"], d["v_new"], kc, vc, d["block_tables"],
                         d["seq_lens"], maxlens[k], wl.scale, out=outs[k], workspace=ws,
                         partition_tokens=part)

    def step(k):
        d = dsteps[k]
        if mode == "append":
            append(k)
            return
        if mode == "positions":
            pa.write_kv_positions(d["k_new"], d["v_new"], d["seq_ids"], d["positions"],
                                  d["block_tables"], kc, vc)
        else:
            pa.write_kv(d["k_new"], d["v_new"], d["slot_mapping"], kc, vc)
        decode(k)

    # The step loop: nothing between the steps' kernels, exactly as a user's
    # loop would issue them (an event between two kernels would stop the
    # programmatic-launch overlap).  The warm-up steps run inside the clock
    # sampler's window, right before the timed ones, so the GPU does not sit
    # idle (and ramp down) between them.
    K = args.steps
    with ClockSampler(device.index or 0) as clocks:
        for w in range(args.warmup):
            step(w % nsteps_wl)
        torch.cuda.synchronize(device)
        if pa.last_device_error() != 0:
            raise RuntimeError("device error flag raised during warm-up")
        rank_barrier()
        torch.cuda.synchronize(device)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for it in range(K):
            step(it % nsteps_wl)
        end.record(stream)
        torch.cuda.synchronize(device)
    rank_barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), device)
    step_bytes_sum = sum(bytes_[it % nsteps_wl]["decode"] + bytes_[it % nsteps_wl]["write"]
                         for it in range(K))
    seqs = wl.num_seqs * K
    value = world * step_bytes_sum / (total_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    err = pa.last_device_error()
    if err != 0:
        raise RuntimeError(f"device error flag {err} raised in the timed region")

    roof = time_decode_calls(append if mode == "append" else decode, nsteps_wl, bytes_, device,
                             stream, peak, peak_kind, total_ms / K, fused=mode == "append")
    if pa.last_device_error() != 0:
        raise RuntimeError("device error flag raised in the roofline block")

    # end to end: host buffers, H2D of the step inputs and D2H of the output
    e2e = run_e2e(args, wl, pa, kc, vc, ws, maxlens, part, device, stream, bytes_, world,
                  shared, fused=mode == "append")

    launches_per_step = []
    for k in range(nsteps_wl):
        n = 1 if wl.steps[k].slot_mapping.numel() and mode != "append" else 0
        n += 1
        need = pa.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, maxlens[k], kc, part)
        n += 1 if need or shared else 0                # the merge
        launches_per_step.append(n)
    launches = sum(launches_per_step[it % nsteps_wl] for it in range(K))
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(wl, args.cpu_seconds, max_reps=100000, gpu_outs=outs,
                          one_core_s=min(5.0, args.cpu_seconds / 2))
    b0 = bytes_[0]
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_name(wl.dtype),
        "data": "synthetic (seeded N(0,1) K/V/q; tables from a shuffled block pool)",
        "config": decode_config(args, wl, world),
        "kernel_config": {
            "partition_tokens": b0["partition"],
            "write": {"append": "inside pa_decode_append", "positions": "pa_write_kv_positions",
                      "slot_mapping": "pa_write_kv"}[mode],
            "decode": ("pa_decode_shared_prefix, automatic mode (%s): %d group(s), "
                       "%s shared blocks"
                       % ("shared blocks read once" if once
                          else "plain decode: reading them once would not pay here",
                          len(wl.prefix_groups), "/".join(str(b) for _, b in wl.prefix_groups))
                       if shared else
                       ("pa_decode_append (the write inside the decode kernel)%s"
                        % ("; %d shared-prefix group(s): the shared-prefix decode's automatic "
                           "mode runs the plain decode on this batch (reading the shared "
                           "blocks once would not pay), which this call is"
                           % len(wl.prefix_groups) if wl.prefix_groups and
                           not args.no_shared_prefix else ""))
                       if mode == "append" else "pa_decode")},
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "decode_tokens_per_s_per_layer": round(world * seqs / (total_ms / 1e3), 1),
        "bytes_per_step": {"unique_kv": b0["unique_kv"], "logical_kv": b0["logical_kv"],
                           "decode": b0["decode"], "write": b0["write"]},
        "roofline": {**roof,
                     "traffic": None if overrides(args) else measured_traffic(args.workload)},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    return result


def time_calls(call, n_distinct, device, stream) -> dict:
    """A library call's time, the way every line's roofline takes it.

    Block: at least ROOF_MIN_CALLS calls and ROOF_MIN_MS milliseconds issued
    back to back on the caller's stream between one pair of CUDA events, with
    nothing between the calls (programmatic-launch overlap intact), so the
    block's time / calls is the mean call.  Clocks are sampled over the block.
    Then ROOF_SAMPLED isolated calls, each between its own pair of events,
    give the median and p10/p90 of one call (an event between calls stops the
    overlap, so these include the launch).  call(c) issues call number c
    (c % n_distinct picks the inputs)."""
    for c in range(3):
        call(c % n_distinct)
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for c in range(10):
        call(c % n_distinct)
    b.record(stream)
    torch.cuda.synchronize(device)
    est = a.elapsed_time(b) / 10                       # one call's time, to size the block
    calls = max(ROOF_MIN_CALLS, math.ceil(ROOF_MIN_MS / max(est, 1e-3)))
    calls = int(max_over_ranks(float(calls), device))  # every rank issues the same block
    with ClockSampler(device.index or 0) as clocks:
        for c in range(10):                           # busy again after the sampler's start
            call(c % n_distinct)
        rank_barrier()
        torch.cuda.synchronize(device)
        a.record(stream)
        for c in range(calls):
            call(c % n_distinct)
        b.record(stream)
        torch.cuda.synchronize(device)
    rank_barrier()
    block_ms = max_over_ranks(a.elapsed_time(b), device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(ROOF_SAMPLED)]
    for c, (e0, e1) in enumerate(evs):
        e0.record(stream)
        call(c % n_distinct)
        e1.record(stream)
    torch.cuda.synchronize(device)
    one = [e0.elapsed_time(e1) for e0, e1 in evs]
    q = statistics.quantiles(one, n=10)
    return {"calls": calls, "block_ms": block_ms, "mean_ms": block_ms / calls,
            "median_ms": statistics.median(one), "p10_ms": q[0], "p90_ms": q[-1],
            "sampled": len(one), "clocks": clocks.summary()}


def roofline_fields(t: dict, what: str, prefix: str, ms_per_step: float) -> dict:
    """The block timing's keys of a line's roofline object."""
    return {"timed_launches": t["calls"], "block_ms": round(t["block_ms"], 3),
            f"{prefix}_ms_mean": round(t["mean_ms"], 5),
            f"{prefix}_ms_median": round(t["median_ms"], 5),
            f"{prefix}_ms_p10": round(t["p10_ms"], 5), f"{prefix}_ms_p90": round(t["p90_ms"], 5),
            "sampled_calls": t["sampled"],
            "per_call_le_step": bool(t["mean_ms"] <= ms_per_step * ROOF_STEP_SLACK),
            "clocks": t["clocks"],
            "how": f"{t['calls']} {what} back to back on the caller's stream between one pair "
                   f"of CUDA events (achieved = their algorithmic work / that time); median "
                   f"and p10/p90 from {t['sampled']} isolated calls, each between its own "
                   f"events"}


def time_decode_calls(decode, nsteps, bytes_, device, stream, peak, peak_kind,
                      ms_per_step, fused: bool = False) -> dict:
    """The roofline figure of the decode call (partition kernel + merge):
    time_calls' block, achieved = the calls' algorithmic bytes / its time.
    With `fused` the call is pa_decode_append, whose bytes include the
    append's (new rows read, cache rows written).  Self-check: the block's
    mean call must not be longer than a whole step of the step loop, within
    ROOF_STEP_SLACK."""
    t = time_calls(decode, nsteps, device, stream)
    keys = ("decode", "write") if fused else ("decode",)
    block_bytes = sum(bytes_[c % nsteps][k] for c in range(t["calls"]) for k in keys)
    achieved = block_bytes / (t["block_ms"] / 1e3) / 1e9
    name = "pa_decode_append" if fused else "pa_decode"
    what = ("partition kernel with the append + merge" if fused
            else "partition kernel + merge")
    return {"bound": "hbm", "kernel": f"{name} call ({what})",
            "achieved": round(achieved, 2), "peak": peak,
            "peak_kind": f"hbm_gbs of {peak_kind}", "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            **roofline_fields(t, f"{name} calls", "decode", ms_per_step)}


def prefill_flops(wl) -> int:
    """4 * D * Hq flops per (query row, visible key): QK^T and PV."""
    st = wl.steps[0]
    total = 0
    for i in range(st.seq_lens.numel()):
        T = int(st.seq_lens[i])
        L = int(st.query_start[i + 1] - st.query_start[i])
        # keys visible from positions T-L .. T-1: sum of (p + 1)
        total += (T * (T + 1) - (T - L) * (T - L + 1)) // 2
    return 4 * wl.head_dim * wl.num_q_heads * total


def run_prefill(args, rank, world, device):
    """Chunked prefill step: pa_write_kv of the chunk tokens + pa_prefill."""
    import paged_kv_cache_109_gb300 as pa
    pa.load_library()
    wl = workloads.make("prefill", **overrides(args))
    st = wl.steps[0]
    kc, vc = wl.k_cache.to(device), wl.v_cache.to(device)
    d = {k: getattr(st, k).to(device) for k in ("q", "k_new", "v_new", "slot_mapping",
                                                "block_tables", "seq_lens", "query_start")}
    out = torch.empty_like(d["q"])
    max_q = int((st.query_start[1:] - st.query_start[:-1]).max())
    max_len = int(st.seq_lens.max())
    stream = torch.cuda.current_stream(device)

    def prefill_call(_=0):
        pa.prefill(d["q"], d["query_start"], kc, vc, d["block_tables"], d["seq_lens"], max_q,
                   max_len, wl.scale, out=out)

    def step():
        pa.write_kv(d["k_new"], d["v_new"], d["slot_mapping"], kc, vc)
        prefill_call()

    K = args.steps
    with ClockSampler(device.index or 0) as clocks:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(device)
        rank_barrier()
        torch.cuda.synchronize(device)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for it in range(K):
            step()
        end.record(stream)
        torch.cuda.synchronize(device)
    rank_barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), device)
    if pa.last_device_error() != 0:
        raise RuntimeError("device error flag raised in the timed region")
    tcalls = time_calls(prefill_call, 1, device, stream)
    flops = prefill_flops(wl)
    by = step_bytes(wl, 0, split_traffic=False)
    step_b = by["decode"] + by["write"]
    tflops = flops * tcalls["calls"] / (tcalls["block_ms"] / 1e3) / 1e12
    peak_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        peak = float(json.load(open(peak_path))["bf16_tflops_sustained"])
        peak_kind = "bf16_tflops_sustained of measured"
    except (OSError, KeyError, ValueError):
        peak, peak_kind = 1700.0, "fallback sustained bf16"
    hbm_peak, _ = measured_peak()
    value = world * K * step_b / (total_ms / 1e3) / 1e9

    # end to end: the chunk's q, new K/V, slots, starts, tables and lengths
    # packed in one page-locked buffer cross in one H2D copy; write + prefill;
    # the output returns in one D2H copy (pipelined as in pipelined_steps)
    names = ("q", "k_new", "v_new", "slot_mapping", "query_start", "block_tables", "seq_lens")
    hbuf, hv = _packed({k: getattr(st, k) for k in names}, pinned=True)
    for k in names:
        hv[k].copy_(getattr(st, k))

    def launch(k, d, o):
        pa.write_kv(d["k_new"], d["v_new"], d["slot_mapping"], kc, vc)
        pa.prefill(d["q"], d["query_start"], kc, vc, d["block_tables"], d["seq_lens"],
                   max_q, max_len, wl.scale, out=o)

    K2 = max(1, min(K, 100))
    e2e_ms = pipelined_steps([(hbuf, hv)], [hv["q"]], launch, K2, device, stream) / K2
    e2e = {"value": round(world * step_b / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hv.values()),
           "d2h_bytes_per_step": hv["q"].numel() * hv["q"].element_size(), "steps": K2,
           "ms_per_step": round(e2e_ms, 5),
           "prefill_tflops": round(flops / (e2e_ms / 1e3) / 1e12, 1),
           "how": "per step: one H2D copy of the packed chunk inputs from pinned memory, "
                  "write + prefill, one D2H copy of the output to pinned memory; copies on "
                  "their own streams, double-buffered, overlapping the neighbouring steps' "
                  "kernels"}
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(wl.dtype),
        "data": "synthetic (seeded N(0,1) K/V/q; tables from a shuffled block pool)",
        "config": prefill_config(args, wl, world),
        "pct_of_hbm_peak": round(100 * value / world / hbm_peak, 2),
        "prefill_tflops": round(tflops, 1),
        "roofline": {"bound": "tensor", "kernel": "pa_prefill call (tcgen05 bf16)",
                     "achieved": round(tflops, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "traffic": None if overrides(args) else measured_traffic("prefill"),
                     "flops_per_call": flops,
                     **roofline_fields(tcalls, "pa_prefill calls", "prefill", total_ms / K)},
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(),
        "cpu_baseline": (time_oracle_prefill(wl, args.cpu_seconds)
                         if rank == 0 and world == 1 and not args.no_cpu_baseline else None),
    }


def run_copy(args, rank, world, device):
    """Block copies: `copy` inside the device pool (HBM read + write), `swap`
    out to page-locked host memory and back (bound by the host link)."""
    import paged_kv_cache_109_gb300 as pa
    pa.load_library()
    stream = torch.cuda.current_stream(device)
    if args.workload == "copy":
        # --num-blocks: a smaller pool (profiling), a quarter of it copied per call
        wl = (workloads.copy_pairs(num_blocks=args.num_blocks, num_pairs=args.num_blocks // 4)
              if args.num_blocks else workloads.copy_pairs())
        kc, vc = wl.k_cache.to(device), wl.v_cache.to(device)
        pairs = wl.pairs.to(device)
        calls = [(kc, vc, kc, vc, pairs)]
        step_bytes_ = wl.copy_bytes()
    else:
        wl = workloads.copy_pairs(num_blocks=8192, num_pairs=2048, fill=True)
        kc, vc = wl.k_cache.to(device), wl.v_cache.to(device)
        host_k = torch.empty((2048,) + tuple(wl.k_cache.shape[1:]), dtype=wl.k_cache.dtype)
        host_k = host_k.pin_memory()
        host_v = torch.empty_like(host_k).pin_memory()
        to_host = torch.stack([wl.pairs[:, 0], torch.arange(2048)], 1).to(device)
        from_host = torch.stack([torch.arange(2048), wl.pairs[:, 1]], 1).to(device)
        calls = [(kc, vc, host_k, host_v, to_host), (host_k, host_v, kc, vc, from_host)]
        step_bytes_ = 2 * wl.copy_bytes()

    def step(_=0):
        for c in calls:
            pa.copy_blocks(*c)

    K = args.steps
    with ClockSampler(device.index or 0) as clocks:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(device)
        rank_barrier()
        torch.cuda.synchronize(device)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for it in range(K):
            step()
        end.record(stream)
        torch.cuda.synchronize(device)
    rank_barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), device)
    if pa.last_device_error() != 0:
        raise RuntimeError("device error flag raised in the timed region")
    tcalls = time_calls(step, 1, device, stream)
    achieved = step_bytes_ * tcalls["calls"] / (tcalls["block_ms"] / 1e3) / 1e9
    value = world * K * step_bytes_ / (total_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    if args.workload == "copy":
        roof = {"bound": "hbm", "kernel": "pa_copy_blocks call", "achieved": round(achieved, 2),
                "peak": peak, "peak_kind": f"hbm_gbs of {peak_kind} (a copy, like this kernel)",
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": None if args.num_blocks else measured_traffic("copy"),
                **roofline_fields(tcalls, "pa_copy_blocks calls", "copy", total_ms / K)}
    else:
        roof = {"bound": "host link", "kernel": "pa_copy_blocks calls (out + in)",
                "achieved": round(achieved, 2), "peak": None, "unit": "GB/s", "frac": None,
                "traffic": None, "note": "device <-> page-locked host copies; no HBM roofline",
                **roofline_fields(tcalls, "swap steps (out + in)", "swap", total_ms / K)}
    # end to end: pairs from pinned host memory each step, one block read back
    host_pairs = [c[4].cpu().pin_memory() for c in calls]
    dev_pairs = [torch.empty_like(c[4]) for c in calls]
    probe = torch.empty(calls[0][2][0].shape, dtype=calls[0][2].dtype).pin_memory()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K2 = max(1, min(K, 200))
    torch.cuda.synchronize(device)
    rank_barrier()
    s2.record(stream)
    for _ in range(K2):
        for c, hp, dp in zip(calls, host_pairs, dev_pairs):
            dp.copy_(hp, non_blocking=True)
            pa.copy_blocks(c[0], c[1], c[2], c[3], dp)
        probe.copy_(calls[-1][2][0], non_blocking=True)
    e2.record(stream)
    torch.cuda.synchronize(device)
    rank_barrier()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2), device) / K2
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) blocks, shuffled pool)",
        "config": copy_config(args, wl, int(calls[0][4].shape[0]), step_bytes_, world),
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "bytes_per_step": step_bytes_,
        "roofline": roof,
        "e2e": {"value": round(world * step_bytes_ / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": sum(h.numel() * 8 for h in host_pairs),
                "d2h_bytes_per_step": probe.numel() * probe.element_size(), "steps": K2},
        "gpu_launches": K * len(calls),
        "clocks": clocks.summary(),
        "cpu_baseline": None,
    }


def _packed(tensors: dict, pinned: bool, device=None):
    """One contiguous buffer holding every tensor (each 256-byte aligned) and
    views of it with the tensors' shapes and dtypes."""
    offs, total = {}, 0
    for name, t in tensors.items():
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = {}
    for name, t in tensors.items():
        nbytes = t.numel() * t.element_size()
        views[name] = buf[offs[name]:offs[name] + nbytes].view(t.dtype).view(t.shape)
    return buf, views


def pipelined_steps(host, outs_like, launch, K, device, stream):
    """Runs K steps end to end from page-locked host buffers the way a serving
    loop overlaps them, and returns the milliseconds between the events that
    bracket them (max over ranks).

    host[k] = (packed pinned buffer, its views) of distinct step k, used for
    step it as k = it % len(host).  Three streams: a copy stream moves step
    it's inputs (one H2D copy) into device slot it % 2, the caller's stream
    waits for them and calls launch(k, device views, device output), and an
    output stream returns the output (one D2H copy) to pinned memory.  So
    step it + 1's input copy and step it - 1's output copy overlap step it's
    kernels.  A slot's inputs are refilled only after the kernels that read
    them have finished, and its output is rewritten only after its copy out.
    Every copy lies inside the timed region."""
    n = len(host)
    slots = [[_packed({nm: t for nm, t in hv.items()}, pinned=False, device=device)
              for _, hv in host] for _ in range(2)]
    outs_d = [[torch.empty_like(o, device=device) for o in outs_like] for _ in range(2)]
    outs_h = [torch.empty_like(o).pin_memory() for o in outs_like]
    cin, cout = torch.cuda.Stream(device), torch.cuda.Stream(device)
    copied, consumed, drained = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def run(steps):
        cin.wait_stream(stream)
        cout.wait_stream(stream)

        def copy_in(it):
            s, k = it % 2, it % n
            with torch.cuda.stream(cin):
                if it >= 2:
                    cin.wait_event(consumed[s])
                slots[s][k][0].copy_(host[k][0], non_blocking=True)
                copied[s].record(cin)

        copy_in(0)
        for it in range(steps):
            s, k = it % 2, it % n
            if it + 1 < steps:
                copy_in(it + 1)
            stream.wait_event(copied[s])
            if it >= 2:
                stream.wait_event(drained[s])
            launch(k, slots[s][k][1], outs_d[s][k])
            consumed[s].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(consumed[s])
                outs_h[k].copy_(outs_d[s][k], non_blocking=True)
                drained[s].record(cout)
        stream.wait_stream(cout)

    run(3)
    torch.cuda.synchronize(device)
    rank_barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    run(K)
    e.record(stream)
    torch.cuda.synchronize(device)
    rank_barrier()
    return max_over_ranks(s.elapsed_time(e), device)


def run_e2e(args, wl, pa, kc, vc, ws, maxlens, part, device, stream, bytes_, world=1,
            shared=False, fused=False):
    """Same step through the public API from pinned host buffers: the step's
    inputs (q, new K/V, slots unless the write is fused, tables, lengths, and
    the shared-prefix groups when used) packed in one page-locked buffer cross
    in one H2D copy; write + decode (one pa_decode_append call when fused);
    the output returns in one D2H copy (pipelined as in pipelined_steps)."""
    names = ("q", "k_new", "v_new", "block_tables", "seq_lens") if fused else \
        ("q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens")
    gnames = ("seq_group", "member_start", "members", "prefix_blocks")
    hgroups = pa.prefix_groups(wl.prefix_groups, wl.num_seqs) if shared else None
    host = []
    for st in wl.steps:
        src = {k: getattr(st, k) for k in names}
        if shared:
            src.update({k: getattr(hgroups, k) for k in gnames})
        hbuf, hv = _packed(src, pinned=True)
        for k, t in src.items():
            hv[k].copy_(t)
        host.append((hbuf, hv))
    n = len(host)
    K = max(1, min(args.steps, 200))

    def launch(k, d, out):
        if fused:
            pa.decode_append(d["q"], d["k_new"], d["v_new"], kc, vc, d["block_tables"],
                             d["seq_lens"], maxlens[k], wl.scale, out=out, workspace=ws,
                             partition_tokens=part)
            return
        pa.write_kv(d["k_new"], d["v_new"], d["slot_mapping"], kc, vc)
        if shared:
            grp = pa.PrefixGroups(d["seq_group"], d["member_start"], d["members"],
                                  d["prefix_blocks"], hgroups.max_group_size,
                                  hgroups.max_prefix_blocks)
            pa.decode_shared_prefix(d["q"], kc, vc, d["block_tables"], d["seq_lens"],
                                    maxlens[k], grp, wl.scale, out=out, workspace=ws,
                                    partition_tokens=part)
        else:
            pa.decode(d["q"], kc, vc, d["block_tables"], d["seq_lens"], maxlens[k], wl.scale,
                      out=out, workspace=ws, partition_tokens=part)

    ms = pipelined_steps(host, [hv["q"] for _, hv in host], launch, K, device, stream)
    total = world * sum(bytes_[it % n]["decode"] + bytes_[it % n]["write"] for it in range(K))
    h2d = sum(t.numel() * t.element_size() for t in host[0][1].values())
    d2h = host[0][1]["q"].numel() * host[0][1]["q"].element_size()
    return {"value": round(total / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "ms_per_step": round(ms / K, 5),
            "how": "per step: one H2D copy of the packed inputs from pinned memory, %s, one "
                   "D2H copy of the output to pinned memory; copies on their own streams, "
                   "double-buffered, overlapping the neighbouring steps' kernels"
                   % ("pa_decode_append (write inside the decode)" if fused
                      else "write + decode")}


def overrides(args) -> dict:
    """Size overrides for profiling smaller cases of a workload."""
    out = {}
    if args.num_seqs:
        out["num_seqs"] = args.num_seqs
        if args.workload == "gqa":
            out["num_shared"] = max(1, args.num_seqs // 4)
    if getattr(args, "prefix_len", 0):
        out["prefix_len"] = args.prefix_len
    if getattr(args, "num_shared", 0):
        out["num_shared"] = args.num_shared
    if args.num_blocks:
        out["num_blocks"] = args.num_blocks
    if args.dtype == "f32":
        out["dtype"] = torch.float32
    if args.head_dim:
        out["head_dim"] = args.head_dim
    if args.block_size:
        # same pool bytes at every block size
        out["block_size"] = args.block_size
        base = {"mha": (8192, 16), "gqa": (65536, 16), "cb": (65536, 16), "long": (16384, 32)}
        nb, bs = base[args.workload]
        if "num_blocks" not in out:
            out["num_blocks"] = nb * bs // args.block_size
    return out


def overrides_json(args) -> dict:
    """overrides() as printed in the JSON line."""
    return {k: dtype_name(v) if isinstance(v, torch.dtype) else v
            for k, v in overrides(args).items()}


def dtype_name(dt) -> str:
    return "f32" if dt == torch.float32 else "bf16"


def run_reference(args, rank, world=1):
    """The oracle as the reference arm: bounded full steps on the host cores.
    Its config is the GPU arm's (the same workload description)."""
    if rank != 0:
        return None
    if args.workload in ("copy", "swap"):
        cpu, wl = time_oracle_copy(args)
        n_pairs = int(wl.pairs.shape[0])
        sb = wl.copy_bytes() if args.workload == "copy" else 2 * wl.copy_bytes()
        return {"impl": "reference", "metric": METRIC, "value": round(cpu["value"], 4),
                "unit": "GB/s", "n_gpus": 0, "steps": cpu["steps"], "warmup": 0,
                "ms_per_step": round(1e3 * cpu["seconds"] / cpu["steps"], 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": copy_config(args, wl, n_pairs, sb, world),
                "cpu_baseline": cpu,
                "e2e": {"value": round(cpu["value"], 4), "unit": "GB/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    wl = workloads.make(args.workload, **overrides(args))
    steps = max(1, args.steps)
    cpu = (time_oracle_prefill(wl, args.cpu_seconds) if args.workload == "prefill"
           else time_oracle(wl, args.cpu_seconds, max_reps=steps))
    return {"impl": "reference", "metric": METRIC, "value": round(cpu["value"], 4),
            "unit": "GB/s", "n_gpus": 0, "steps": cpu["steps"], "warmup": 0,
            "ms_per_step": round(1e3 * cpu["seconds"] / cpu["steps"], 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": (prefill_config(args, wl, world) if args.workload == "prefill"
                       else decode_config(args, wl, world)),
            "cpu_baseline": cpu,
            "e2e": {"value": round(cpu["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def make_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="long")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="smaller batch (profiling); the JSON line then has no traffic")
    ap.add_argument("--num-blocks", type=int, default=0, help="smaller block pool (profiling)")
    ap.add_argument("--block-size", type=int, default=0,
                    help="block-size sweep: tokens per block (pool bytes kept constant)")
    ap.add_argument("--prefix-len", type=int, default=0,
                    help="gqa: tokens of the shared prefix (whole blocks; 512 by default)")
    ap.add_argument("--num-shared", type=int, default=0,
                    help="gqa: sequences that share the prefix (32 by default)")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="decode a workload with shared-prefix groups (gqa) with the plain "
                         "pa_decode instead of pa_decode_shared_prefix")
    ap.add_argument("--write", choices=["auto", "append", "slot_mapping", "positions"],
                    default="auto",
                    help="how a decode step writes its new tokens: inside the decode call "
                         "(append: steps that add one token per sequence at its last "
                         "position), pa_write_kv with a slot mapping, or "
                         "pa_write_kv_positions; auto = append where the steps allow it")
    ap.add_argument("--positions", action="store_true",
                    help="same as --write positions")
    ap.add_argument("--dtype", choices=["bf16", "f32"], default="bf16",
                    help="cache and q dtype of a decode workload (f32 runs the CUDA-core "
                         "decode kernel)")
    ap.add_argument("--head-dim", type=int, default=0,
                    help="head dim of a decode workload (other than 64 and 128: the "
                         "CUDA-core decode kernel)")
    return ap


def main():
    ap = make_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload in ("copy", "swap", "prefill") and (args.dtype != "bf16" or args.head_dim):
        ap.error("--dtype and --head-dim apply to the decode workloads")
    if args.workload != "gqa" and (args.prefix_len or args.num_shared):
        ap.error("--prefix-len and --num-shared apply to the gqa workload")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    runner = {"copy": run_copy, "swap": run_copy, "prefill": run_prefill}.get(args.workload,
                                                                          run_ours)
    res = runner(args, rank, world, device)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
