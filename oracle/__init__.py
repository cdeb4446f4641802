"""Plain fp64 CPU oracle for paged-attention decode and the slot-mapping write.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are its only users.  The CUDA library and its
Python binding never import it, and the two share no code.

The arithmetic lives in ``pa_oracle.c`` (compiled with gcc into
``liboracle.so``); this module only marshals arrays.  What it follows:

* "vLLM PagedAttention: from memory fragmentation to slot mapping" §2-§4:
  block counts, tail waste, and the logical -> physical -> slot formula.
* "PagedAttention" (LLM glossary), contiguous vs page-table section: gather K/V
  by table into contiguous rows, then plain softmax attention; query heads are
  grouped with ``repeat_interleave`` (head h reads kv head h // (Hq/Hkv)).
* "vLLM source walkthrough: PagedAttention and Continuous Batching" §1.8 (V2
  partitions + reduce) and the paper notes' 10-token blockwise example:
  per-partition (acc, m, l) and a log-sum-exp merge.
* The cache write: each new token's K/V rows go to ``slot_mapping[j]``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (OpenMP when available).  Returns the path."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *extra_flags, "-o", out, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    target = path or _LIB
    if path is None and (not os.path.exists(target)
                         or os.path.getmtime(target) < os.path.getmtime(_SRC)):
        build()
    lib = ctypes.CDLL(target)
    P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_blocks_needed.argtypes = [I64, I32]
    lib.oracle_blocks_needed.restype = I64
    lib.oracle_tail_waste.argtypes = [I64, I32]
    lib.oracle_tail_waste.restype = I64
    lib.oracle_slot.argtypes = [P, I32, I64]
    lib.oracle_slot.restype = I64
    lib.oracle_attend.argtypes = [P, P, P, I64, I32, D, P]
    lib.oracle_attend.restype = None
    lib.oracle_decode.argtypes = [P, P, P, ctypes.c_int, I32, I32, I32, I32, P, I32, P,
                                  I32, I32, D, P, I64, P]
    lib.oracle_decode.restype = I64
    lib.oracle_decode_partials.argtypes = [P, P, P, ctypes.c_int, I32, I32, I32, I32, P,
                                           I32, P, I32, I32, D, I32, I32, P, P, P]
    lib.oracle_decode_partials.restype = I64
    lib.oracle_merge.argtypes = [I32, P, P, P, I32, P]
    lib.oracle_merge.restype = None
    lib.oracle_write_kv.argtypes = [P, P, P, I64, P, P, I32, I32, I32, I32, I32]
    lib.oracle_write_kv.restype = I64
    lib.oracle_prefill.argtypes = [P, P, P, P, ctypes.c_int, I32, I32, I32, I32, P, I32, P,
                                   I32, I32, D, P]
    lib.oracle_prefill.restype = I64
    lib.oracle_copy_blocks.argtypes = [P, P, I32, P, P, I32, P, I64, I64]
    lib.oracle_copy_blocks.restype = I64
    lib.oracle_slots_from_positions.argtypes = [P, P, I64, P, I32, I32, I32, P]
    lib.oracle_slots_from_positions.restype = None
    lib.oracle_set_threads.argtypes = [I32]
    lib.oracle_set_threads.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = I32
    if path is None:
        _lib = lib
    return lib


@contextlib.contextmanager
def using(path: str):
    """Route every call in the block through the library at ``path`` (used by
    the tests that check the pins reject deliberately broken oracle builds)."""
    global _lib
    saved = _lib
    _lib = load(path)
    try:
        yield _lib
    finally:
        _lib = saved


# ---- array marshalling ----------------------------------------------------

def _as_array(x):
    """Host numpy view of a CPU tensor or array.  bf16 tensors become uint16
    bit patterns (the oracle widens them exactly); returns (array, dtype code)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.is_cuda:
                raise ValueError("oracle inputs must be host tensors")
            x = x.contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            return x.numpy(), None
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    return a, None


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(x):
    a, _ = _as_array(x)
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(x):
    a, _ = _as_array(x)
    return np.ascontiguousarray(a, dtype=np.int64)


# ---- addressing -----------------------------------------------------------

def blocks_needed(num_tokens: int, block_size: int) -> int:
    return int(load().oracle_blocks_needed(num_tokens, block_size))


def tail_waste(num_tokens: int, block_size: int) -> int:
    return int(load().oracle_tail_waste(num_tokens, block_size))


def physical_slot(table, block_size: int, position: int) -> int:
    t = _i32(table)
    return int(load().oracle_slot(_ptr(t), block_size, position))


# ---- attention ------------------------------------------------------------

def attend(q, K, V, scale: float) -> np.ndarray:
    """Dense softmax attention of one query row q[D] over K[T,D], V[T,D] (fp64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    out = np.zeros(q.shape[-1], dtype=np.float64)
    load().oracle_attend(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.shape[-1], scale, _ptr(out))
    return out


def _cache_geometry(k_cache):
    nb, hkv, bs, d = (int(s) for s in k_cache.shape)
    return nb, hkv, bs, d


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale: float, pairs=None,
           threads: int | None = None) -> np.ndarray:
    """fp64 out[N, Hq, D] of single-query attention read through block tables.

    q is [N, Hq, D]; caches are [num_blocks, Hkv, B, D] (fp32 or bf16, same
    dtype as q); block_tables int32 [N, max_blocks]; seq_lens int32 [N].
    ``pairs`` (optional [P, 2] of (seq, q_head)) limits the work to those rows;
    the others are NaN.
    """
    qa, dt = _as_array(q)
    ka, dk = _as_array(k_cache)
    va, dv = _as_array(v_cache)
    if dt is None or dt != dk or dt != dv:
        raise ValueError("q and caches must share one dtype (float32 or bfloat16)")
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    n, hq, d = (int(s) for s in q.shape)
    nb, hkv, bs, dd = _cache_geometry(k_cache)
    if dd != d or hq % hkv:
        raise ValueError("shape mismatch")
    out = np.full((n, hq, d), np.nan, dtype=np.float64)
    lib = load()
    if threads:
        lib.oracle_set_threads(threads)
    if pairs is None:
        pp, npairs = None, 0
    else:
        pa = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        pp, npairs = _ptr(pa), pa.shape[0]
    bad = lib.oracle_decode(_ptr(qa), _ptr(ka), _ptr(va), dt, nb, bs, hkv, d, _ptr(bt),
                            bt.shape[1], _ptr(sl), n, hq, scale, pp, npairs, _ptr(out))
    if bad:
        raise ValueError(f"{bad} (seq, head) rows met an invalid block-table entry")
    return out


def prefill(q, query_start_loc, k_cache, v_cache, block_tables, seq_lens,
            scale: float) -> np.ndarray:
    """fp64 out[total_q, Hq, D] of causal multi-query attention: sequence i's
    rows query_start_loc[i]..query_start_loc[i+1] are its last positions."""
    qa, dt = _as_array(q)
    ka, dk = _as_array(k_cache)
    va, dv = _as_array(v_cache)
    if dt is None or dt != dk or dt != dv:
        raise ValueError("q and caches must share one dtype (float32 or bfloat16)")
    qs = _i32(query_start_loc)
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    total, hq, d = (int(s) for s in q.shape)
    nb, hkv, bs, _ = _cache_geometry(k_cache)
    n = sl.shape[0]
    if qs.shape[0] != n + 1 or qs[-1] != total:
        raise ValueError("query_start_loc must have num_seqs + 1 entries ending at total_q")
    out = np.full((total, hq, d), np.nan, dtype=np.float64)
    bad = load().oracle_prefill(_ptr(qa), _ptr(qs), _ptr(ka), _ptr(va), dt, nb, bs, hkv, d,
                                _ptr(bt), bt.shape[1], _ptr(sl), n, hq, scale, _ptr(out))
    if bad:
        raise ValueError(f"{bad} (row, head) results met an invalid length or table entry")
    return out


def decode_partials(q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                    partition_tokens: int, max_parts: int | None = None):
    """Per-partition (m, l, acc) in natural-log units; arrays are
    [N, Hq, max_parts] and [N, Hq, max_parts, D]; unused cells are NaN."""
    qa, dt = _as_array(q)
    ka, _ = _as_array(k_cache)
    va, _ = _as_array(v_cache)
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    n, hq, d = (int(s) for s in q.shape)
    nb, hkv, bs, _ = _cache_geometry(k_cache)
    if max_parts is None:
        max_parts = max(1, -(-int(sl.max(initial=0)) // partition_tokens))
    m = np.full((n, hq, max_parts), np.nan)
    l = np.full((n, hq, max_parts), np.nan)
    acc = np.full((n, hq, max_parts, d), np.nan)
    bad = load().oracle_decode_partials(_ptr(qa), _ptr(ka), _ptr(va), dt, nb, bs, hkv, d,
                                        _ptr(bt), bt.shape[1], _ptr(sl), n, hq, scale,
                                        partition_tokens, max_parts, _ptr(m), _ptr(l),
                                        _ptr(acc))
    if bad:
        raise ValueError(f"{bad} (seq, head) rows met an invalid block-table entry")
    return m, l, acc


def merge(m, l, acc) -> np.ndarray:
    """Log-sum-exp merge of partials m[P], l[P], acc[P, D] into out[D]."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    out = np.zeros(acc.shape[-1], dtype=np.float64)
    load().oracle_merge(m.shape[0], _ptr(m), _ptr(l), _ptr(acc), acc.shape[-1], _ptr(out))
    return out


# ---- cache write ----------------------------------------------------------

def write_kv(k, v, slot_mapping, k_cache, v_cache) -> int:
    """Scatter k, v [n_tok, Hkv, D] into the caches (host tensors or arrays,
    modified in place) at slot_mapping [n_tok]; returns the count of slots at
    or beyond num_blocks * B (skipped)."""
    for c in (k_cache, v_cache):
        contiguous = c.is_contiguous() if hasattr(c, "is_contiguous") else c.flags.c_contiguous
        if not contiguous:
            raise ValueError("caches must be contiguous host buffers (written in place)")
    ka, _ = _as_array(k)
    va, _ = _as_array(v)
    sm = _i64(slot_mapping)
    kc, _ = _as_array(k_cache)
    vc, _ = _as_array(v_cache)
    nb, hkv, bs, d = _cache_geometry(k_cache)
    return int(load().oracle_write_kv(_ptr(ka), _ptr(va), _ptr(sm), sm.shape[0], _ptr(kc),
                                      _ptr(vc), nb, bs, hkv, d, ka.itemsize))


def copy_blocks(src_k, src_v, dst_k, dst_v, pairs) -> int:
    """Copy whole blocks src -> dst for each (src, dst) row of ``pairs`` (in
    order), from the source caches into the destination caches (host, written
    in place; may be the same tensors).  Returns the count of rejected pairs."""
    for c in (dst_k, dst_v):
        contiguous = c.is_contiguous() if hasattr(c, "is_contiguous") else c.flags.c_contiguous
        if not contiguous:
            raise ValueError("destination caches must be contiguous host buffers")
    sk, _ = _as_array(src_k)
    sv, _ = _as_array(src_v)
    dk, _ = _as_array(dst_k)
    dv, _ = _as_array(dst_v)
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    block_bytes = sk.itemsize * int(np.prod(src_k.shape[1:]))
    return int(load().oracle_copy_blocks(_ptr(sk), _ptr(sv), int(src_k.shape[0]), _ptr(dk),
                                         _ptr(dv), int(dst_k.shape[0]), _ptr(pr), pr.shape[0],
                                         block_bytes))


def slots_from_positions(seq_ids, positions, block_tables, block_size: int) -> np.ndarray:
    """int64 slots of tokens given by (sequence id, position) through the tables."""
    si = _i32(seq_ids)
    po = _i32(positions)
    bt = _i32(block_tables)
    out = np.empty(si.shape[0], dtype=np.int64)
    load().oracle_slots_from_positions(_ptr(si), _ptr(po), si.shape[0], _ptr(bt), bt.shape[0],
                                       bt.shape[1], block_size, _ptr(out))
    return out


def set_threads(n: int) -> None:
    load().oracle_set_threads(n)


def max_threads() -> int:
    return int(load().oracle_max_threads())
