"""Paged-attention decode for GB300: Python binding of libpa.so.

Every function here marshals tensors into the C ABI declared in
``include/pa.h``; all computation runs in the library's CUDA kernels.  There
is no CPU path: every call raises ``ImportError`` when ``libpa.so`` has not
been built, and the calls only accept CUDA tensors.

    import paged_kv_cache_109_gb300 as pa
    pa.write_kv(k, v, slot_mapping, k_cache, v_cache)
    out = pa.decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len)
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from ._build import LIB as LIBRARY_PATH
from ._build import build
from .block_pool import BlockPool, SharedTailWrite

__all__ = ["write_kv", "write_kv_positions", "copy_blocks", "decode", "decode_append",
           "decode_shared_prefix", "prefix_groups", "PrefixGroups", "decode_shared_prefix_workspace_bytes",
           "decode_shared_prefix_mode", "prefill",
           "decode_workspace_bytes", "decode_partition_tokens",
           "decode_path", "last_device_error", "PaError", "build", "BlockPool",
           "SharedTailWrite", "LIBRARY_PATH", "load_library", "CacheDesc"]

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)
PA_F32, PA_BF16 = 0, 1
DEVERR_TABLE_ENTRY, DEVERR_SEQ_LEN, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_BLOCK_PAIR = 1, 2, 4, 8, 16
DEVERR_GROUP = 32
SHARED_AUTO, SHARED_ONCE, SHARED_PLAIN = 0, 1, 2


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_str(status)} (status {status})")


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libpa.so (built in-tree by ``build()``); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    target = path or LIBRARY_PATH
    if not os.path.exists(target):
        raise ImportError(f"{target} is not built; run paged_kv_cache_109_gb300.build()")
    lib = ctypes.CDLL(target)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    DP = ctypes.POINTER(CacheDesc)
    lib.pa_write_kv.argtypes = [P, P, P, I32, P, P, DP, P]
    lib.pa_write_kv.restype = ctypes.c_int
    lib.pa_write_kv_positions.argtypes = [P, P, P, P, I32, P, I32, I32, P, P, DP, P]
    lib.pa_write_kv_positions.restype = ctypes.c_int
    lib.pa_copy_blocks.argtypes = [P, P, I32, P, P, I32, P, I32, DP, P]
    lib.pa_copy_blocks.restype = ctypes.c_int
    lib.pa_prefill.argtypes = [P, P, I32, I32, P, P, P, I32, P, I32, I32, I32, ctypes.c_float,
                               P, DP, P]
    lib.pa_prefill.restype = ctypes.c_int
    lib.pa_decode_partition_tokens.argtypes = [I32, I32, I32, DP]
    lib.pa_decode_partition_tokens.restype = I32
    lib.pa_decode_workspace_bytes.argtypes = [I32, I32, I32, I32, DP]
    lib.pa_decode_workspace_bytes.restype = SZ
    lib.pa_decode.argtypes = [P, P, P, P, I32, P, I32, I32, I32, ctypes.c_float, I32, P, P, SZ,
                              DP, P]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_decode_append.argtypes = [P, P, P, P, P, P, I32, P, I32, I32, I32, ctypes.c_float,
                                     I32, P, P, SZ, DP, P]
    lib.pa_decode_append.restype = ctypes.c_int
    lib.pa_decode_shared_prefix_workspace_bytes.argtypes = [I32, I32, I32, I32, I32, DP]
    lib.pa_decode_shared_prefix_workspace_bytes.restype = SZ
    lib.pa_decode_shared_prefix.argtypes = [P, P, P, P, I32, P, I32, I32, I32, ctypes.c_float,
                                            I32, P, P, P, P, I32, I32, I32, I32, P, P, SZ, DP,
                                            P]
    lib.pa_decode_shared_prefix_mode.argtypes = [I32, I32, I32, DP]
    lib.pa_decode_shared_prefix_mode.restype = I32
    lib.pa_decode_shared_prefix.restype = ctypes.c_int
    lib.pa_decode_path.argtypes = [I32, DP]
    lib.pa_decode_path.restype = I32
    lib.pa_status_str.argtypes = [ctypes.c_int]
    lib.pa_status_str.restype = ctypes.c_char_p
    lib.pa_last_device_error.argtypes = []
    lib.pa_last_device_error.restype = I32
    lib.pa_check_wait_timeout.argtypes = [I32, I32, ctypes.c_int64, P]
    lib.pa_check_wait_timeout.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _status_str(status: int) -> str:
    try:
        return load_library().pa_status_str(status).decode()
    except ImportError:
        return "unknown"


# ---- marshalling helpers ----------------------------------------------------

_DTYPES = {torch.float32: PA_F32, torch.bfloat16: PA_BF16}


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    if k_cache.dim() != 4:
        raise ValueError("caches are [num_blocks, num_kv_heads, block_size, head_dim]")
    if k_cache.dtype not in _DTYPES:
        raise ValueError(f"unsupported cache dtype {k_cache.dtype}")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d, _DTYPES[k_cache.dtype])


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _dev(*ts: torch.Tensor) -> None:
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _dev_or_pinned(*ts: torch.Tensor) -> None:
    for t in ts:
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("tensors must be on a CUDA device or in page-locked host memory")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PaError(status, where)


# ---- public calls -------------------------------------------------------------

def write_kv(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Scatter k, v [n_tok, Hkv, D] into the caches at slot_mapping [n_tok] (int64).
    k, v and slot_mapping may be page-locked host tensors: the kernel reads them
    over the host link."""
    _dev(k_cache, v_cache)
    _dev_or_pinned(k, v, slot_mapping)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise ValueError("k, v and caches must share one dtype")
    desc = cache_desc(k_cache)
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache shapes differ")
    n = slot_mapping.numel()
    if k.shape != (n, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
        raise ValueError(f"k, v must be [{n}, {desc.num_kv_heads}, {desc.head_dim}]")
    st = load_library().pa_write_kv(_ptr(k), _ptr(v), _ptr(slot_mapping), n, _ptr(k_cache),
                                    _ptr(v_cache), ctypes.byref(desc), _stream(stream))
    _check(st, "pa_write_kv")


def write_kv_positions(k, v, seq_ids, positions, block_tables, k_cache, v_cache,
                       stream=None) -> None:
    """Scatter k, v [n_tok, Hkv, D] to the slots of (seq_ids[j], positions[j])
    through block_tables [N, max_blocks]; slots are computed on the device.
    Everything but the caches may be page-locked host memory."""
    _dev(k_cache, v_cache)
    _dev_or_pinned(k, v, seq_ids, positions, block_tables)
    for t in (seq_ids, positions, block_tables):
        if t.dtype != torch.int32:
            raise ValueError("seq_ids, positions and block_tables must be int32")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise ValueError("k, v and caches must share one dtype")
    desc = cache_desc(k_cache)
    n = seq_ids.numel()
    if positions.numel() != n or k.shape != (n, desc.num_kv_heads, desc.head_dim) \
            or v.shape != k.shape:
        raise ValueError("k, v, seq_ids and positions disagree on the token count")
    st = load_library().pa_write_kv_positions(
        _ptr(k), _ptr(v), _ptr(seq_ids), _ptr(positions), n, _ptr(block_tables),
        block_tables.shape[0], block_tables.shape[1], _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(desc), _stream(stream))
    _check(st, "pa_write_kv_positions")


def copy_blocks(src_k, src_v, dst_k, dst_v, pairs, stream=None) -> None:
    """Copy whole blocks src -> dst for each row (src, dst) of ``pairs``
    (int64 [n, 2]).  Caches may be device tensors or pinned host tensors
    (swap space); the destination may be the source (copy-on-write)."""
    _dev_or_pinned(src_k, src_v, dst_k, dst_v, pairs)
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [n, 2]")
    if tuple(src_k.shape[1:]) != tuple(dst_k.shape[1:]) or src_k.dtype != dst_k.dtype:
        raise ValueError("source and destination caches differ in block geometry")
    desc = cache_desc(src_k)
    st = load_library().pa_copy_blocks(
        _ptr(src_k), _ptr(src_v), src_k.shape[0], _ptr(dst_k), _ptr(dst_v), dst_k.shape[0],
        _ptr(pairs), pairs.shape[0], ctypes.byref(desc), _stream(stream))
    _check(st, "pa_copy_blocks")


def decode_partition_tokens(num_seqs: int, num_q_heads: int, max_seq_len: int,
                            k_cache) -> int:
    desc = k_cache if isinstance(k_cache, CacheDesc) else cache_desc(k_cache)
    return int(load_library().pa_decode_partition_tokens(num_seqs, num_q_heads, max_seq_len,
                                                         ctypes.byref(desc)))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, max_seq_len: int, k_cache,
                           partition_tokens: int = 0) -> int:
    desc = k_cache if isinstance(k_cache, CacheDesc) else cache_desc(k_cache)
    return int(load_library().pa_decode_workspace_bytes(num_seqs, num_q_heads, max_seq_len,
                                                        partition_tokens, ctypes.byref(desc)))


def decode_path(num_q_heads: int, k_cache) -> int:
    desc = k_cache if isinstance(k_cache, CacheDesc) else cache_desc(k_cache)
    return int(load_library().pa_decode_path(num_q_heads, ctypes.byref(desc)))


def decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len: int,
           scale: float | None = None, out=None, workspace=None, partition_tokens: int = 0,
           stream=None) -> torch.Tensor:
    """Single-query paged attention; returns out [N, Hq, D] in the cache dtype.

    ``max_seq_len`` is a host-side upper bound of ``seq_lens`` (no device
    read-back).  ``workspace`` (uint8, device) is allocated if not given and
    split-K needs one.  q, block_tables, seq_lens and out may be page-locked
    host tensors, read and written by the kernels over the host link; a
    missing ``out`` is allocated on the caches' device.
    """
    _dev(k_cache, v_cache)
    _dev_or_pinned(q, block_tables, seq_lens)
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    desc = cache_desc(k_cache)
    n, hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, device=k_cache.device)
    _dev_or_pinned(out)
    need = decode_workspace_bytes(n, hq, max_seq_len, desc, partition_tokens)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_cache.device)
    if workspace is not None:
        _dev(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().pa_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), n, max_seq_len, hq, float(scale), partition_tokens, _ptr(out),
        _ptr(workspace), ws_bytes, ctypes.byref(desc), _stream(stream))
    _check(st, "pa_decode")
    return out


def decode_append(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                  max_seq_len: int, scale: float | None = None, out=None, workspace=None,
                  partition_tokens: int = 0, stream=None) -> torch.Tensor:
    """One decode step in one call: sequence i's newest token, at position
    seq_lens[i] - 1, takes the rows k_new[i], v_new[i] ([N, Hkv, D]) in both
    caches, then the decode runs as ``decode`` does.  Caches and output equal
    ``write_kv_positions`` (positions seq_lens - 1) followed by ``decode``,
    bit for bit; on the TMA decode kernel the write is fused into it."""
    _dev(k_cache, v_cache)
    _dev_or_pinned(q, k_new, v_new, block_tables, seq_lens)
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    if k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype \
            or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_new, v_new and caches must share one dtype")
    desc = cache_desc(k_cache)
    n, hq, d = q.shape
    if k_new.shape != (n, desc.num_kv_heads, desc.head_dim) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new, v_new must be [{n}, {desc.num_kv_heads}, {desc.head_dim}]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, device=k_cache.device)
    _dev_or_pinned(out)
    need = decode_workspace_bytes(n, hq, max_seq_len, desc, partition_tokens)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_cache.device)
    if workspace is not None:
        _dev(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().pa_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), n, max_seq_len, hq, float(scale),
        partition_tokens, _ptr(out), _ptr(workspace), ws_bytes, ctypes.byref(desc),
        _stream(stream))
    _check(st, "pa_decode_append")
    return out


class PrefixGroups:
    """The groups of a shared-prefix decode as the C ABI takes them: int32
    tensors ``seq_group`` [num_seqs] (group of each sequence, -1 for none),
    ``member_start`` [num_groups + 1], ``members`` and ``prefix_blocks``
    [num_groups], with the host bounds ``max_group_size`` and
    ``max_prefix_blocks``."""

    def __init__(self, seq_group, member_start, members, prefix_blocks, max_group_size: int,
                 max_prefix_blocks: int):
        self.seq_group = seq_group
        self.member_start = member_start
        self.members = members
        self.prefix_blocks = prefix_blocks
        self.max_group_size = int(max_group_size)
        self.max_prefix_blocks = int(max_prefix_blocks)

    @property
    def num_groups(self) -> int:
        return int(self.prefix_blocks.numel())

    def to(self, device) -> "PrefixGroups":
        return PrefixGroups(self.seq_group.to(device), self.member_start.to(device),
                            self.members.to(device), self.prefix_blocks.to(device),
                            self.max_group_size, self.max_prefix_blocks)


def prefix_groups(groups, num_seqs: int, device=None) -> PrefixGroups:
    """PrefixGroups from a list of (member sequence ids, shared leading
    blocks), e.g. ``BlockPool.shared_prefix_groups``; groups of fewer than
    two members are dropped."""
    groups = [(list(map(int, m)), int(b)) for m, b in groups if len(m) >= 2]
    seq_group = [-1] * num_seqs
    starts, members, blocks = [0], [], []
    for k, (mem, b) in enumerate(groups):
        for i in mem:
            seq_group[i] = k
        members += mem
        starts.append(len(members))
        blocks.append(b)

    def i32(x):
        return torch.tensor(x, dtype=torch.int32, device=device)

    return PrefixGroups(i32(seq_group), i32(starts), i32(members), i32(blocks),
                        max((len(m) for m, _ in groups), default=0),
                        max(blocks, default=0))


def decode_shared_prefix_workspace_bytes(num_seqs: int, num_q_heads: int, max_seq_len: int,
                                         max_prefix_blocks: int, k_cache,
                                         partition_tokens: int = 0) -> int:
    desc = k_cache if isinstance(k_cache, CacheDesc) else cache_desc(k_cache)
    return int(load_library().pa_decode_shared_prefix_workspace_bytes(
        num_seqs, num_q_heads, max_seq_len, max_prefix_blocks, partition_tokens,
        ctypes.byref(desc)))


def decode_shared_prefix_mode(num_q_heads: int, max_prefix_blocks: int, k_cache,
                              mode: int = SHARED_AUTO) -> int:
    """1 when decode_shared_prefix reads the shared blocks once per row tile
    for these arguments, 0 when it runs the plain decode."""
    desc = k_cache if isinstance(k_cache, CacheDesc) else cache_desc(k_cache)
    return int(load_library().pa_decode_shared_prefix_mode(num_q_heads, max_prefix_blocks,
                                                           mode, ctypes.byref(desc)))


def decode_shared_prefix(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len: int,
                         groups: PrefixGroups, scale: float | None = None, out=None,
                         workspace=None, partition_tokens: int = 0, mode: int = SHARED_AUTO,
                         stream=None) -> torch.Tensor:
    """``decode`` for a batch whose ``groups`` of sequences share leading
    blocks: the same result, with each group's shared blocks read once per
    kv head and row tile instead of once per member (``mode``: SHARED_ONCE,
    SHARED_PLAIN, or SHARED_AUTO to choose by the expected saving)."""
    _dev(k_cache, v_cache)
    _dev_or_pinned(q, block_tables, seq_lens, groups.seq_group, groups.member_start,
                   groups.members, groups.prefix_blocks)
    for t in (block_tables, seq_lens, groups.seq_group, groups.member_start, groups.members,
              groups.prefix_blocks):
        if t.dtype != torch.int32:
            raise ValueError("tables, lengths and group arrays must be int32")
    desc = cache_desc(k_cache)
    n, hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, device=k_cache.device)
    _dev_or_pinned(out)
    need = decode_shared_prefix_workspace_bytes(n, hq, max_seq_len, groups.max_prefix_blocks,
                                                desc, partition_tokens)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_cache.device)
    if workspace is not None:
        _dev(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().pa_decode_shared_prefix(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), n, max_seq_len, hq, float(scale), partition_tokens,
        _ptr(groups.seq_group), _ptr(groups.member_start), _ptr(groups.members),
        _ptr(groups.prefix_blocks), groups.num_groups, groups.max_group_size,
        groups.max_prefix_blocks, mode, _ptr(out), _ptr(workspace), ws_bytes,
        ctypes.byref(desc), _stream(stream))
    _check(st, "pa_decode_shared_prefix")
    return out


def last_device_error() -> int:
    """PA_DEVERR_* bits raised since the last call (synchronises the device)."""
    return int(load_library().pa_last_device_error())


def check_wait_timeout(expected: int, arrivals: int, limit_cycles: int, stream=None) -> None:
    """Runs the bounded-wait check: an mbarrier needing `expected` arrivals
    gets `arrivals`, and one CTA waits for it for at most `limit_cycles`
    clocks (PA_DEVERR_TIMEOUT when it gives up; read last_device_error())."""
    st = load_library().pa_check_wait_timeout(expected, arrivals, limit_cycles,
                                              _stream(stream))
    _check(st, "pa_check_wait_timeout")


def prefill(q, query_start_loc, k_cache, v_cache, block_tables, seq_lens, max_q_len: int,
            max_seq_len: int, scale: float | None = None, out=None, stream=None):
    """Causal multi-query attention over the paged cache: sequence i's packed
    rows query_start_loc[i]..query_start_loc[i+1] are its last positions.
    Returns out [total_q, Hq, D] in the cache dtype.  Everything but the
    caches may be page-locked host memory (read and written over the host
    link); a missing ``out`` is allocated on the caches' device."""
    _dev(k_cache, v_cache)
    _dev_or_pinned(q, query_start_loc, block_tables, seq_lens)
    for t in (query_start_loc, block_tables, seq_lens):
        if t.dtype != torch.int32:
            raise ValueError("query_start_loc, block_tables and seq_lens must be int32")
    desc = cache_desc(k_cache)
    total, hq, d = q.shape
    if query_start_loc.numel() != seq_lens.numel() + 1:
        raise ValueError("query_start_loc must have num_seqs + 1 entries")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, device=k_cache.device)
    _dev_or_pinned(out)
    st = load_library().pa_prefill(
        _ptr(q), _ptr(query_start_loc), total, max_q_len, _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), seq_lens.numel(), max_seq_len,
        hq, float(scale), _ptr(out), ctypes.byref(desc), _stream(stream))
    _check(st, "pa_prefill")
    return out
