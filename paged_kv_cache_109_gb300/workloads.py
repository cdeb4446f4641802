"""Seeded synthetic inputs for the decode and cache-write calls.

This module draws random numbers and builds block tables through the host
``BlockPool``; it holds none of the attention arithmetic.  Tests feed what it
returns both to the CUDA library and to the CPU oracle, and the benchmark
times the CUDA library on it.  Everything is produced on the host (CPU
tensors); callers copy to the device.

Workloads (shapes follow the serving examples on the pages):

``tiny``  fp32, the glossary page's worked example: lengths 10 and 7, B=4,
          Hq=4, Hkv=2, D=8, 7 physical blocks, tables [[5,1,6],[5,3,-1]],
          block 5 holding the shared 4-token prefix (V prefix = 0.5 * K
          prefix), torch seed 53 drawn in that page's script order.
``mha``   bf16, N=32, Hq=Hkv=32, D=128, B=16, T ~ U[128, 2048], tables taken
          from a shuffled free list over an 8192-block pool.
``gqa``   bf16, N=128, Hq=32, Hkv=8, D=128, B=16, T ~ round(lognormal(ln 1024,
          1.0)) capped at 8192; 32 sequences share one 512-token prefix
          (32 physical blocks with ref_cnt 32); 65536-block shuffled pool.
``long``  bf16, N=4, T=131072, Hq=64, Hkv=8, D=128, B=32; one permutation of
          a 16384-block pool split into four 4096-entry tables.
``cb``    bf16 continuous batching, N=256, Hq=32, Hkv=8, D=128, B=16,
          T0 ~ U[1, 4096], 65536-block pool; each of 10 steps appends one
          token to every sequence and a 2048-token chunk to one seeded pick
          (2304 writes per step), growing tables when a tail block fills.

Every decode step first writes the step's new tokens (the last position of
each decoding sequence), then attends over all T_i positions including them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

from .block_pool import BlockPool, slot_of

_CHUNKS = 16


def normal(shape, seed: int, tag: int, dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, 1) float32 draws cast to ``dtype``; deterministic for (seed, tag)
    whatever the thread count (16 fixed PCG64 streams, one per chunk)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    streams = np.random.SeedSequence([int(seed), int(tag)]).spawn(_CHUNKS)
    bounds = [n * i // _CHUNKS for i in range(_CHUNKS + 1)]

    def fill(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            np.random.default_rng(streams[i]).standard_normal(hi - lo, dtype=np.float32,
                                                              out=out[lo:hi])

    with ThreadPoolExecutor(max(1, min(_CHUNKS, os.cpu_count() or 1))) as ex:
        list(ex.map(fill, range(_CHUNKS)))
    return torch.from_numpy(out).view(*shape).to(dtype)


@dataclass
class Step:
    q: torch.Tensor              # [N, Hq, D]
    k_new: torch.Tensor          # [n_tok, Hkv, D]
    v_new: torch.Tensor          # [n_tok, Hkv, D]
    slot_mapping: torch.Tensor   # [n_tok] int64
    block_tables: torch.Tensor   # [N, width] int32, -1 padded
    seq_lens: torch.Tensor       # [N] int32, lengths after this step's writes
    seq_ids: torch.Tensor = None     # [n_tok] int32: sequence of each new token
    positions: torch.Tensor = None   # [n_tok] int32: its position in that sequence
    query_start: torch.Tensor = None  # [N + 1] int32: query rows per sequence (prefill)


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_blocks: int
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    k_cache: torch.Tensor        # history before the first step, [nb, Hkv, B, D]
    v_cache: torch.Tensor
    steps: list[Step]
    seed: int
    stats: dict = field(default_factory=dict)
    # groups of sequences sharing leading blocks (member ids, shared blocks),
    # from the pool's tables and reference counts (BlockPool.shared_prefix_groups)
    prefix_groups: list = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return int(self.steps[0].seq_lens.numel())   # q has one row per query token

    @property
    def max_seq_len(self) -> int:
        return max(int(s.seq_lens.max()) for s in self.steps)

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()

    def kv_bytes_read(self, step: int = 0) -> int:
        """K+V bytes of the valid tokens of one decode (each sequence counted)."""
        t = int(self.steps[step].seq_lens.to(torch.int64).sum())
        return t * 2 * self.num_kv_heads * self.head_dim * self.elem_bytes

    def describe(self) -> dict:
        return {"workload": self.name, "dtype": str(self.dtype).replace("torch.", ""),
                "num_seqs": self.num_seqs, "num_q_heads": self.num_q_heads,
                "num_kv_heads": self.num_kv_heads, "head_dim": self.head_dim,
                "block_size": self.block_size, "num_blocks": self.num_blocks,
                "steps": len(self.steps), "seed": self.seed, **self.stats}


def _fill_history(pool: BlockPool, hkv: int, d: int, dtype, seed: int):
    """Caches with N(0,1) rows in every block a table references, zeros elsewhere."""
    shape = (pool.num_blocks, hkv, pool.block_size, d)
    k_cache = torch.zeros(shape, dtype=dtype)
    v_cache = torch.zeros(shape, dtype=dtype)
    used = sorted({b for t in pool.tables.values() for b in t})
    if used:
        idx = torch.tensor(used, dtype=torch.int64)
        k_cache[idx] = normal((len(used), hkv, pool.block_size, d), seed, 1, dtype)
        v_cache[idx] = normal((len(used), hkv, pool.block_size, d), seed, 2, dtype)
    return k_cache, v_cache


def _decode_step(pool: BlockPool, seqs, hq: int, hkv: int, d: int, width: int, dtype,
                 seed: int, tag: int) -> Step:
    """One decode step: the new token of each sequence is its last position."""
    n = len(seqs)
    lens = [pool.lengths[s] for s in seqs]
    slots = [pool.slot(s, lens[i] - 1) for i, s in enumerate(seqs)]
    return Step(q=normal((n, hq, d), seed, tag, dtype),
                k_new=normal((n, hkv, d), seed, tag + 1, dtype),
                v_new=normal((n, hkv, d), seed, tag + 2, dtype),
                slot_mapping=torch.tensor(slots, dtype=torch.int64),
                block_tables=torch.tensor(pool.table_rows(seqs, width), dtype=torch.int32),
                seq_lens=torch.tensor(lens, dtype=torch.int32),
                seq_ids=torch.arange(n, dtype=torch.int32),
                positions=torch.tensor(lens, dtype=torch.int32) - 1)


def _stats(pool: BlockPool, seqs) -> dict:
    return {"unique_blocks": pool.unique_blocks(), "live_tokens": pool.live_tokens(),
            "block_utilization": round(pool.utilization(), 6),
            "logical_tokens": sum(pool.lengths[s] for s in seqs)}


# ---- the worked example ---------------------------------------------------

def tiny() -> Workload:
    """Glossary page worked example; draws follow that page's script order:
    prefix [2,4,8]; K tails [2,6,8], [2,3,8]; V tails [2,6,8], [2,3,8]; q [2,4,1,8]."""
    hq, hkv, d, bs, lengths = 4, 2, 8, 4, (10, 7)
    g = torch.Generator().manual_seed(53)
    prefix = torch.randn(hkv, 4, d, generator=g, dtype=torch.float32)
    k_tails = [torch.randn(hkv, n - 4, d, generator=g) for n in lengths]
    v_tails = [torch.randn(hkv, n - 4, d, generator=g) for n in lengths]
    q = torch.randn(2, hq, 1, d, generator=g, dtype=torch.float32).reshape(2, hq, d)
    contiguous_k = [torch.cat((prefix, t), 1) for t in k_tails]        # [Hkv, T, D]
    contiguous_v = [torch.cat((prefix * 0.5, t), 1) for t in v_tails]
    tables = [[5, 1, 6], [5, 3, -1]]
    # sequence 0 writes all 10 positions; sequence 1 reuses block 5 for its
    # first 4 positions and writes positions 4..6 into its own block 3
    written = [(0, p) for p in range(10)] + [(1, p) for p in range(4, 7)]
    slots = [slot_of(tables[s], bs, p) for s, p in written]
    k_new = torch.stack([contiguous_k[s][:, p] for s, p in written])   # [13, Hkv, D]
    v_new = torch.stack([contiguous_v[s][:, p] for s, p in written])
    step = Step(q=q, k_new=k_new, v_new=v_new,
                slot_mapping=torch.tensor(slots, dtype=torch.int64),
                block_tables=torch.tensor(tables, dtype=torch.int32),
                seq_lens=torch.tensor(lengths, dtype=torch.int32),
                seq_ids=torch.tensor([s_ for s_, _ in written], dtype=torch.int32),
                positions=torch.tensor([p_ for _, p_ in written], dtype=torch.int32))
    zeros = torch.zeros(7, hkv, bs, d, dtype=torch.float32)
    wl = Workload("tiny", torch.float32, 7, bs, hq, hkv, d, 1.0 / math.sqrt(d),
                  zeros, zeros.clone(), [step], 53,
                  {"unique_blocks": 4, "live_tokens": 13})
    wl.contiguous_k = contiguous_k
    wl.contiguous_v = contiguous_v
    return wl


# ---- serving-shaped workloads ---------------------------------------------

def mha(num_seqs=32, num_heads=32, head_dim=128, block_size=16, min_len=128,
        max_len=2048, num_blocks=8192, seed=2, dtype=torch.bfloat16) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_len, max_len + 1, size=num_seqs)
    pool = BlockPool(num_blocks, block_size, rng.permutation(num_blocks))
    seqs = list(range(num_seqs))
    for s in seqs:
        pool.add(s, int(lens[s]))
    width = pool.blocks_for(max_len)
    kc, vc = _fill_history(pool, num_heads, head_dim, dtype, seed)
    step = _decode_step(pool, seqs, num_heads, num_heads, head_dim, width, dtype, seed, 10)
    return Workload("mha", dtype, num_blocks, block_size, num_heads, num_heads, head_dim,
                    1.0 / math.sqrt(head_dim), kc, vc, [step], seed, _stats(pool, seqs))


def gqa(num_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        median_len=1024, sigma=1.0, max_len=8192, num_shared=32, prefix_len=512,
        num_blocks=65536, seed=3, dtype=torch.bfloat16) -> Workload:
    rng = np.random.default_rng(seed)
    lens = np.minimum(np.rint(rng.lognormal(math.log(median_len), sigma, size=num_seqs)),
                      max_len).astype(np.int64)
    sharers = set(rng.choice(num_seqs, size=num_shared, replace=False).tolist()) \
        if num_shared else set()
    lens = [max(int(t), prefix_len + 1) if s in sharers else max(int(t), 1)
            for s, t in enumerate(lens)]
    pool = BlockPool(num_blocks, block_size, rng.permutation(num_blocks))
    if sharers:
        pool.add("prefix", prefix_len)
    seqs = list(range(num_seqs))
    for s in seqs:
        if s in sharers:
            pool.add(s, lens[s], prefix_of="prefix", prefix_tokens=prefix_len)
        else:
            pool.add(s, lens[s])
    if sharers:
        pool.release("prefix")
    width = pool.blocks_for(max(max_len, max(lens)))
    kc, vc = _fill_history(pool, num_kv_heads, head_dim, dtype, seed)
    step = _decode_step(pool, seqs, num_q_heads, num_kv_heads, head_dim, width, dtype,
                        seed, 10)
    wl = Workload("gqa", dtype, num_blocks, block_size, num_q_heads, num_kv_heads, head_dim,
                  1.0 / math.sqrt(head_dim), kc, vc, [step], seed, _stats(pool, seqs))
    wl.stats["shared_seqs"] = sorted(sharers)
    wl.stats["prefix_ref_cnt"] = (pool.ref_cnt[pool.tables[min(sharers)][0]]
                                  if sharers else 0)
    wl.prefix_groups = pool.shared_prefix_groups(seqs)
    return wl


def long(num_seqs=4, seq_len=131072, num_q_heads=64, num_kv_heads=8, head_dim=128,
         block_size=32, num_blocks=None, seed=4, dtype=torch.bfloat16) -> Workload:
    per_seq = -(-seq_len // block_size)
    num_blocks = num_blocks or per_seq * num_seqs
    rng = np.random.default_rng(seed)
    pool = BlockPool(num_blocks, block_size, rng.permutation(num_blocks))
    seqs = list(range(num_seqs))
    for s in seqs:
        pool.add(s, seq_len)
    kc, vc = _fill_history(pool, num_kv_heads, head_dim, dtype, seed)
    step = _decode_step(pool, seqs, num_q_heads, num_kv_heads, head_dim, per_seq, dtype,
                        seed, 10)
    return Workload("long", dtype, num_blocks, block_size, num_q_heads, num_kv_heads,
                    head_dim, 1.0 / math.sqrt(head_dim), kc, vc, [step], seed,
                    _stats(pool, seqs))


def cb(num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
       max_len0=4096, chunk=2048, num_steps=10, num_blocks=65536, seed=5,
       dtype=torch.bfloat16) -> Workload:
    """Continuous-batching steps: every sequence decodes one token; one seeded
    pick also takes a prefill chunk, written before its decode token."""
    rng = np.random.default_rng(seed)
    lens0 = rng.integers(1, max_len0 + 1, size=num_seqs)
    pool = BlockPool(num_blocks, block_size, rng.permutation(num_blocks))
    seqs = list(range(num_seqs))
    for s in seqs:
        pool.add(s, int(lens0[s]))
    kc, vc = _fill_history(pool, num_kv_heads, head_dim, dtype, seed)
    width = pool.blocks_for(max_len0 + num_steps * (chunk + 1))
    steps = []
    for k in range(num_steps):
        pick = int(rng.integers(num_seqs))
        slots, tok_seq, tok_pos = [], [], []
        for s in seqs:
            start = pool.lengths[s]
            count = chunk + 1 if s == pick else 1
            pool.grow(s, count)
            slots.extend(pool.slots(s, start, count))
            tok_seq.extend([s] * count)
            tok_pos.extend(range(start, start + count))
        n_tok = len(slots)
        tag = 100 + 10 * k
        steps.append(Step(q=normal((num_seqs, num_q_heads, head_dim), seed, tag, dtype),
                          k_new=normal((n_tok, num_kv_heads, head_dim), seed, tag + 1, dtype),
                          v_new=normal((n_tok, num_kv_heads, head_dim), seed, tag + 2, dtype),
                          slot_mapping=torch.tensor(slots, dtype=torch.int64),
                          block_tables=torch.tensor(pool.table_rows(seqs, width),
                                                    dtype=torch.int32),
                          seq_lens=torch.tensor([pool.lengths[s] for s in seqs],
                                                dtype=torch.int32),
                          seq_ids=torch.tensor(tok_seq, dtype=torch.int32),
                          positions=torch.tensor(tok_pos, dtype=torch.int32)))
    return Workload("cb", dtype, num_blocks, block_size, num_q_heads, num_kv_heads, head_dim,
                    1.0 / math.sqrt(head_dim), kc, vc, steps, seed, _stats(pool, seqs))


def prefill(num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
            max_len0=4096, chunk=2048, num_blocks=65536, seed=7,
            dtype=torch.bfloat16) -> Workload:
    """Chunked prefill: every sequence has a seeded history T0 ~ U[1, max_len0]
    and takes a chunk of `chunk` new tokens; the step writes the chunk's K/V,
    then attends causally from each chunk token (q rows = the chunk)."""
    rng = np.random.default_rng(seed)
    lens0 = rng.integers(1, max_len0 + 1, size=num_seqs)
    pool = BlockPool(num_blocks, block_size, rng.permutation(num_blocks))
    seqs = list(range(num_seqs))
    for s in seqs:
        pool.add(s, int(lens0[s]))
    kc, vc = _fill_history(pool, num_kv_heads, head_dim, dtype, seed)
    slots, tok_seq, tok_pos, qs = [], [], [], [0]
    for s in seqs:
        start = pool.lengths[s]
        pool.grow(s, chunk)
        slots.extend(pool.slots(s, start, chunk))
        tok_seq.extend([s] * chunk)
        tok_pos.extend(range(start, start + chunk))
        qs.append(qs[-1] + chunk)
    n_tok = len(slots)
    width = pool.blocks_for(max_len0 + chunk)
    step = Step(q=normal((n_tok, num_q_heads, head_dim), seed, 10, dtype),
                k_new=normal((n_tok, num_kv_heads, head_dim), seed, 11, dtype),
                v_new=normal((n_tok, num_kv_heads, head_dim), seed, 12, dtype),
                slot_mapping=torch.tensor(slots, dtype=torch.int64),
                block_tables=torch.tensor(pool.table_rows(seqs, width), dtype=torch.int32),
                seq_lens=torch.tensor([pool.lengths[s] for s in seqs], dtype=torch.int32),
                seq_ids=torch.tensor(tok_seq, dtype=torch.int32),
                positions=torch.tensor(tok_pos, dtype=torch.int32),
                query_start=torch.tensor(qs, dtype=torch.int32))
    return Workload("prefill", dtype, num_blocks, block_size, num_q_heads, num_kv_heads,
                    head_dim, 1.0 / math.sqrt(head_dim), kc, vc, [step], seed,
                    _stats(pool, seqs))


@dataclass
class CopyWorkload:
    """Whole-block copies inside one pool: num_pairs disjoint (src, dst) pairs
    over a shuffled pool (the copy-on-write / swap copy)."""
    name: str
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    pairs: torch.Tensor          # int64 [num_pairs, 2]
    seed: int

    @property
    def block_bytes(self) -> int:
        return self.k_cache[0].numel() * self.k_cache.element_size()

    def copy_bytes(self) -> int:
        """Bytes one call moves: K and V blocks, each read once and written once."""
        return 2 * 2 * self.pairs.shape[0] * self.block_bytes


def copy_pairs(num_blocks=65536, num_pairs=8192, num_kv_heads=8, head_dim=128, block_size=16,
               seed=6, dtype=torch.bfloat16, fill=True) -> CopyWorkload:
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_blocks)
    pairs = torch.tensor(np.stack([perm[:num_pairs], perm[num_pairs:2 * num_pairs]], 1),
                         dtype=torch.int64)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    if fill:
        k = normal(shape, seed, 1, dtype)
        v = normal(shape, seed, 2, dtype)
    else:
        k = torch.zeros(shape, dtype=dtype)
        v = torch.zeros(shape, dtype=dtype)
    return CopyWorkload("copy", k, v, pairs, seed)


BUILDERS = {"tiny": tiny, "mha": mha, "gqa": gqa, "long": long, "cb": cb, "prefill": prefill}


def make(name: str, **overrides) -> Workload:
    return BUILDERS[name](**overrides)
