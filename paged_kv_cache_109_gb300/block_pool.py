"""Host-side block pool: the control plane that produces block tables and
slot mappings for the device calls.  It is not on the hot path.

Behaviour follows the pages:

* free blocks sit in a FIFO queue; a request takes blocks from the front and
  a released block goes to the back ("vLLM PagedAttention: from memory
  fragmentation to slot mapping" §4 timeline; "vLLM source walkthrough" §1.4);
* taking blocks is all-or-nothing: when the pool cannot cover the request,
  ``MemoryError`` is raised and no state changes (same page, §4: a failed
  grow must leave the free list and the tables untouched);
* every block carries a reference count; a sequence that shares another's
  full prefix blocks increments their counts, and a block returns to the free
  queue only when its count drops to zero ("vLLM source walkthrough" §1.6;
  first page §5);
* position p of a sequence lives in slot table[p // B] * B + p % B
  (first page §3).

A write into a shared, partly filled tail block is refused with
``SharedTailWrite`` until ``copy_on_write`` has given the sequence a private
copy; ``copy_on_write``, ``swap_out`` and ``swap_in`` return the block pairs
the device copy (``pa_copy_blocks``) must move.
"""
from __future__ import annotations

from collections import deque
from typing import Hashable, Iterable, Sequence


class SharedTailWrite(RuntimeError):
    """A write would land in a block whose reference count is above one."""


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Iterable[int] | None = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.free_queue: deque[int] = deque(order)
        self.ref_cnt = [0] * self.num_blocks
        self.tables: dict[Hashable, list[int]] = {}
        self.lengths: dict[Hashable, int] = {}

    # -- capacity ------------------------------------------------------------
    def blocks_for(self, num_tokens: int) -> int:
        return -(-int(num_tokens) // self.block_size)

    @property
    def num_free(self) -> int:
        return len(self.free_queue)

    def _take_fresh(self, count: int) -> list[int]:
        if count < 0:
            raise ValueError("negative block count")
        if count > len(self.free_queue):
            raise MemoryError(f"need {count} blocks, {len(self.free_queue)} free")
        fresh = [self.free_queue.popleft() for _ in range(count)]
        for b in fresh:
            self.ref_cnt[b] = 1
        return fresh

    # -- sequence lifecycle --------------------------------------------------
    def add(self, seq: Hashable, num_tokens: int, prefix_of: Hashable | None = None,
            prefix_tokens: int = 0) -> list[int]:
        """Register ``seq`` with ``num_tokens`` tokens.  With ``prefix_of``,
        the first ``prefix_tokens`` (a multiple of B, at most both lengths)
        reuse that sequence's full blocks instead of fresh ones."""
        if seq in self.tables:
            raise KeyError(f"sequence {seq!r} already present")
        shared: list[int] = []
        if prefix_of is not None:
            if prefix_tokens % self.block_size:
                raise ValueError("a shared prefix must cover whole blocks")
            if prefix_tokens > min(num_tokens, self.lengths[prefix_of]):
                raise ValueError("prefix longer than one of the sequences")
            shared = self.tables[prefix_of][: prefix_tokens // self.block_size]
        fresh = self._take_fresh(self.blocks_for(num_tokens) - len(shared))
        for b in shared:
            self.ref_cnt[b] += 1
        self.tables[seq] = list(shared) + fresh
        self.lengths[seq] = int(num_tokens)
        return self.tables[seq]

    def grow(self, seq: Hashable, new_tokens: int) -> list[int]:
        """Append ``new_tokens`` positions; returns the blocks taken for them."""
        old_len = self.lengths[seq]
        table = self.tables[seq]
        if new_tokens > 0 and old_len % self.block_size:
            tail = table[-1]
            if self.ref_cnt[tail] > 1:
                raise SharedTailWrite(f"block {tail} is shared (ref_cnt {self.ref_cnt[tail]})")
        extra = self.blocks_for(old_len + new_tokens) - len(table)
        fresh = self._take_fresh(max(extra, 0))
        table.extend(fresh)
        self.lengths[seq] = old_len + int(new_tokens)
        return fresh

    def fork(self, parent: Hashable, child: Hashable) -> list[int]:
        """``child`` starts as a copy of ``parent`` sharing every block,
        including a partly filled tail (parallel sampling / beam search
        branches: nxmr.cn article §4.1; paper notes, copy-on-write)."""
        if child in self.tables:
            raise KeyError(f"sequence {child!r} already present")
        table = list(self.tables[parent])
        for b in table:
            self.ref_cnt[b] += 1
        self.tables[child] = table
        self.lengths[child] = self.lengths[parent]
        return table

    def copy_on_write(self, seq: Hashable) -> tuple[int, int] | None:
        """Before ``seq`` appends into a partly filled tail block that other
        sequences share, give it a private copy: take a fresh block, point the
        table at it and drop one reference to the old block (nxmr.cn article
        §4.2).  Returns the (old, new) pair whose K/V the device must copy,
        or None when the tail is full or already private."""
        n = self.lengths[seq]
        table = self.tables[seq]
        if n % self.block_size == 0 or not table:
            return None
        tail = table[-1]
        if self.ref_cnt[tail] <= 1:
            return None
        fresh = self._take_fresh(1)[0]
        self.ref_cnt[tail] -= 1
        table[-1] = fresh
        return tail, fresh

    def append_step(self, seqs: Sequence[Hashable]) -> list[tuple[int, int]]:
        """One decode step: each of ``seqs`` appends one position, the token
        ``pa_decode_append`` then writes at its new length - 1.  Per sequence,
        in order (nxmr.cn article §4.2, the append rule): a full tail block is
        followed by a fresh block; a partly filled tail that other sequences
        share is first replaced by a private copy (``copy_on_write``);
        otherwise the token goes into the tail as it is.  Returns the
        (old, new) block pairs the device must copy (``pa_copy_blocks``)
        before the step.  All or nothing: when the pool cannot cover every
        sequence's blocks, ``MemoryError`` is raised and no state changes."""
        if len(set(seqs)) != len(seqs):
            raise ValueError("a sequence appears twice in one step")
        # dry run: blocks needed, with the reference drops of earlier copies
        drops: dict[int, int] = {}
        need = 0
        for seq in seqs:
            n, table = self.lengths[seq], self.tables[seq]
            if n % self.block_size == 0:
                need += 1
            elif self.ref_cnt[table[-1]] - drops.get(table[-1], 0) > 1:
                need += 1
                drops[table[-1]] = drops.get(table[-1], 0) + 1
        if need > len(self.free_queue):
            raise MemoryError(f"need {need} blocks, {len(self.free_queue)} free")
        pairs = []
        for seq in seqs:
            pair = self.copy_on_write(seq)
            if pair is not None:
                pairs.append(pair)
            self.grow(seq, 1)
        return pairs

    def swap_out(self, seq: Hashable, host: "BlockPool") -> list[tuple[int, int]]:
        """Move ``seq``'s blocks to the host pool (paper notes, swapping):
        returns the (device block, host block) pairs to copy; the device blocks
        go back to this pool's free queue.  Every block must be private to
        ``seq``.  All-or-nothing: MemoryError leaves both pools unchanged."""
        table = self.tables[seq]
        if any(self.ref_cnt[b] != 1 for b in table):
            raise SharedTailWrite(f"sequence {seq!r} shares blocks; it cannot be swapped alone")
        host_blocks = host._take_fresh(len(table))
        host.tables[seq] = host_blocks
        host.lengths[seq] = self.lengths[seq]
        pairs = list(zip(table, host_blocks))
        self.release(seq)
        return pairs

    def swap_in(self, seq: Hashable, host: "BlockPool") -> list[tuple[int, int]]:
        """Bring ``seq`` back from the host pool: returns the (host block,
        device block) pairs to copy; the host blocks are released."""
        host_table = host.tables[seq]
        fresh = self._take_fresh(len(host_table))
        self.tables[seq] = fresh
        self.lengths[seq] = host.lengths[seq]
        pairs = list(zip(host_table, fresh))
        host.release(seq)
        return pairs

    def release(self, seq: Hashable) -> list[int]:
        """Drop ``seq``; blocks whose count reaches zero rejoin the free queue
        in table order.  Returns those blocks."""
        table = self.tables.pop(seq)
        del self.lengths[seq]
        freed = []
        for b in table:
            self.ref_cnt[b] -= 1
            if self.ref_cnt[b] < 0:
                raise AssertionError(f"block {b} released more often than acquired")
            if self.ref_cnt[b] == 0:
                freed.append(b)
        self.free_queue.extend(freed)
        return freed

    # -- addressing ----------------------------------------------------------
    def slot(self, seq: Hashable, position: int) -> int:
        if not 0 <= position < self.lengths[seq]:
            raise IndexError(position)
        return slot_of(self.tables[seq], self.block_size, position)

    def slots(self, seq: Hashable, start: int, count: int) -> list[int]:
        return [self.slot(seq, p) for p in range(start, start + count)]

    def table_rows(self, seqs: Sequence[Hashable], width: int | None = None) -> list[list[int]]:
        """Tables of ``seqs`` padded with -1 to ``width`` entries."""
        width = max((len(self.tables[s]) for s in seqs), default=0) if width is None else width
        rows = []
        for s in seqs:
            t = self.tables[s]
            if len(t) > width:
                raise ValueError(f"table of {s!r} has {len(t)} entries > width {width}")
            rows.append(t + [-1] * (width - len(t)))
        return rows

    def shared_prefix_groups(self, seqs: Sequence[Hashable]) -> list[tuple[list[int], int]]:
        """Groups of the batch ``seqs`` whose tables start with the same
        shared blocks, for the shared-prefix decode: a list of (member
        positions in ``seqs``, leading blocks every member holds in common).
        Sequences group by their first block when its reference count is
        above one (a prefix added with ``prefix_of`` or a ``fork``); a
        group's count is the longest run of leading entries all its members'
        tables agree on.  A sequence alone in its group is left out."""
        by_first: dict[int, list[int]] = {}
        for idx, s in enumerate(seqs):
            t = self.tables[s]
            if t and self.ref_cnt[t[0]] > 1:
                by_first.setdefault(t[0], []).append(idx)
        groups = []
        for members in by_first.values():
            if len(members) < 2:
                continue
            rows = [self.tables[seqs[m]] for m in members]
            k, n = 0, min(len(r) for r in rows)
            while k < n and all(r[k] == rows[0][k] for r in rows):
                k += 1
            groups.append((members, k))
        return groups

    # -- statistics ----------------------------------------------------------
    def unique_blocks(self) -> int:
        return sum(1 for c in self.ref_cnt if c > 0)

    def live_tokens(self) -> int:
        """Distinct token positions held: a shared prefix block counts once."""
        seen: dict[int, int] = {}
        for s, t in self.tables.items():
            n = self.lengths[s]
            for lb, b in enumerate(t):
                filled = min(self.block_size, n - lb * self.block_size)
                seen[b] = max(seen.get(b, 0), filled)
        return sum(seen.values())

    def utilization(self) -> float:
        """live tokens / (allocated blocks * B)  (nxmr.cn article §5.2)."""
        used = self.unique_blocks()
        return self.live_tokens() / (used * self.block_size) if used else 1.0


def slot_of(table: Sequence[int], block_size: int, position: int) -> int:
    """slot = table[p // B] * B + p % B for one position of one table."""
    physical = int(table[position // block_size])
    if physical < 0:
        raise IndexError(f"position {position} maps to a padding entry")
    return physical * block_size + position % block_size
