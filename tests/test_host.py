"""Host-side logic: the block pool against the pages' allocator examples, and
the seeded workloads' structure.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import workloads
from paged_kv_cache_109_gb300.block_pool import BlockPool, SharedTailWrite, slot_of
from tests.conftest import golden


def test_allocator_timeline():
    g = golden("allocator_timeline.json")
    pool = BlockPool(g["num_blocks"], g["block_size"])
    for op in g["ops"]:
        if op["op"] == "add":
            pool.add(op["seq"], op["tokens"])
        elif op["op"] == "grow":
            pool.grow(op["seq"], op["tokens"])
        else:
            pool.release(op["seq"])
        if "table" in op:
            assert pool.tables[op["seq"]] == op["table"], op
        assert list(pool.free_queue) == op["free"], op
    sc = g["slot_check"]
    assert pool.slot(sc["seq"], sc["position"]) == sc["slot"]
    before = (list(pool.free_queue), {k: v[:] for k, v in pool.tables.items()},
              dict(pool.lengths), list(pool.ref_cnt))
    with pytest.raises(MemoryError):
        pool.grow(g["failed_grow"]["seq"], g["failed_grow"]["tokens"])
    after = (list(pool.free_queue), {k: v[:] for k, v in pool.tables.items()},
             dict(pool.lengths), list(pool.ref_cnt))
    assert before == after


def test_refcount_example():
    g = golden("refcount.json")
    bs = g["block_size"]
    pool = BlockPool(8, bs)
    a = pool.add("A", g["A_tokens"])
    b = pool.add("B", g["B_tokens"], prefix_of="A", prefix_tokens=g["shared_prefix_tokens"])
    names = {a[0]: "b0", a[1]: "b1", a[2]: "b2", b[2]: "b3"}
    order = [a[0], a[1], a[2], b[2]]
    assert [pool.ref_cnt[x] for x in order] == g["ref_after_both"]
    freed = pool.release("A")
    assert [pool.ref_cnt[x] for x in order] == g["ref_after_A_ends"]
    assert [names[x] for x in freed] == g["freed_when_A_ends"]
    freed = pool.release("B")
    assert [pool.ref_cnt[x] for x in order] == g["ref_after_B_ends"]
    assert sorted(names[x] for x in freed) == sorted(g["freed_when_B_ends"])
    assert pool.num_free == 8


def test_shared_prefix_counts():
    g = golden("shared_prefix.json")
    pool = BlockPool(g["num_blocks"], g["block_size"], free_order=[5, 1, 6, 3, 0, 2, 4])
    pool.add(0, g["lengths"][0])
    pool.add(1, g["lengths"][1], prefix_of=0, prefix_tokens=4)
    assert pool.table_rows([0, 1], 3) == g["tables"]
    assert pool.unique_blocks() == g["unique_blocks"]
    assert pool.live_tokens() == g["live_tokens"]
    allocated = pool.unique_blocks() * g["block_size"]
    assert allocated == g["allocated_slots"]
    assert allocated - pool.live_tokens() == g["internal_fragmentation_slots"]
    unshared = sum(pool.blocks_for(t) for t in g["lengths"]) * g["block_size"]
    assert unshared == g["unshared_slots"]
    assert unshared - allocated == g["prefix_sharing_saved_slots"]


def test_shared_tail_write_refused():
    pool = BlockPool(8, 4)
    pool.add("A", 8)
    pool.add("B", 8, prefix_of="A", prefix_tokens=8)
    pool.grow("B", 1)               # tail of B was full: a fresh block, fine
    pool.add("C", 6)
    pool.add("D", 4, prefix_of="C", prefix_tokens=4)
    pool.release("C")
    pool.grow("D", 0)
    with pytest.raises(SharedTailWrite):
        BlockPool.grow(_shared_partial_tail_pool(), "Y", 1)


def _shared_partial_tail_pool():
    pool = BlockPool(6, 4)
    pool.add("X", 4)
    pool.add("Y", 4, prefix_of="X", prefix_tokens=4)
    pool.lengths["Y"] = 3           # tail block of Y partly filled and shared
    return pool


def test_pool_slots_agree_with_oracle_addressing():
    """The host's slot mapping (an input to the write call) agrees with the
    oracle's own addressing on every position of a random pool."""
    rng = np.random.default_rng(0)
    pool = BlockPool(300, 16, rng.permutation(300))
    for s in range(12):
        pool.add(s, int(rng.integers(1, 300)))
    for s in range(12):
        table = pool.tables[s]
        for p in range(pool.lengths[s]):
            assert pool.slot(s, p) == oracle.physical_slot(table, 16, p)
    for case in golden("addressing.json")["cases"]:
        for p, sl in zip(case["positions"], case["slots"]):
            assert slot_of(case["table"], case["block_size"], p) == sl


def test_sizing_figures():
    g = golden("sizing.json")
    kv = g["kv_per_token"]
    per_layer = 2 * kv["kv_heads"] * kv["head_dim"] * kv["elem_bytes"]
    assert per_layer * kv["layers"] == kv["bytes_per_token"]
    assert kv["bytes_per_token"] * 2048 == kv["tokens_2048_bytes"]
    assert kv["bytes_per_token"] * kv["tokens_4k"] * kv["requests"] == kv["batch_bytes"]
    mb = g["max_num_blocks"]
    assert mb["kv_bytes"] // (mb["block_size"] * mb["bytes_per_token"]) == mb["blocks"]
    tw = g["tail_waste"]
    for bs, pct in zip(tw["block_sizes"], tw["approx_waste_pct"]):
        # about half a block per request
        assert abs(100 * (bs / 2) / tw["mean_len"] - pct) <= 0.5


def test_utilization_tracks_half_block_rule():
    rng = np.random.default_rng(1)
    for bs in (16, 32, 64):
        pool = BlockPool(20000, bs)
        lens = rng.integers(1, 1000, size=400)
        for s, t in enumerate(lens):
            pool.add(s, int(t))
        approx = 1 - bs / (2 * lens.mean())
        assert abs(pool.utilization() - approx) < 0.02


def test_tiny_workload_matches_worked_example():
    g = golden("shared_prefix.json")
    wl = workloads.tiny()
    st = wl.steps[0]
    assert st.slot_mapping.tolist() == g["derived_slot_mapping"]["slots"]
    assert st.block_tables.tolist() == g["tables"]
    assert st.seq_lens.tolist() == g["lengths"]
    assert st.q.shape == (2, 4, 8) and st.k_new.shape == (13, 2, 8)
    # the script's draw order: regenerating with seed 53 gives the same prefix
    gen = torch.Generator().manual_seed(53)
    prefix = torch.randn(2, 4, 8, generator=gen)
    assert torch.equal(wl.contiguous_k[0][:, :4], prefix)
    assert torch.equal(wl.contiguous_v[1][:, :4], prefix * 0.5)


def _check_step_invariants(wl, step):
    bs = wl.block_size
    n_tok = step.slot_mapping.numel()
    slots = step.slot_mapping.tolist()
    assert len(set(slots)) == n_tok, "duplicate slots"
    assert min(slots) >= 0 and max(slots) < wl.num_blocks * bs
    bt = step.block_tables
    for i, t in enumerate(step.seq_lens.tolist()):
        need = -(-t // bs)
        assert (bt[i, :need] >= 0).all() and (bt[i, need:] == -1).all()
        assert step.block_tables.shape[1] * bs >= t


def test_mha_small_structure():
    wl = workloads.mha(num_seqs=6, num_heads=4, head_dim=32, min_len=20, max_len=90,
                       num_blocks=64)
    st = wl.steps[0]
    _check_step_invariants(wl, st)
    assert st.k_new.shape == (6, 4, 32)
    # the new token is each sequence's last position
    for i, t in enumerate(st.seq_lens.tolist()):
        assert int(st.slot_mapping[i]) == oracle.physical_slot(st.block_tables[i], 16, t - 1)
    # determinism
    wl2 = workloads.mha(num_seqs=6, num_heads=4, head_dim=32, min_len=20, max_len=90,
                        num_blocks=64)
    assert torch.equal(wl.k_cache, wl2.k_cache) and torch.equal(st.q, wl2.steps[0].q)


def test_gqa_small_shared_prefix():
    wl = workloads.gqa(num_seqs=16, num_q_heads=8, num_kv_heads=2, head_dim=32,
                       median_len=100, max_len=400, num_shared=4, prefix_len=64,
                       num_blocks=512)
    st = wl.steps[0]
    _check_step_invariants(wl, st)
    shared = wl.stats["shared_seqs"]
    assert len(shared) == 4 and wl.stats["prefix_ref_cnt"] == 4
    rows = st.block_tables[shared, :4]
    assert (rows == rows[0]).all()
    # no write lands in a shared prefix block
    prefix_blocks = set(rows[0].tolist())
    for s in st.slot_mapping.tolist():
        assert s // 16 not in prefix_blocks
    assert wl.stats["unique_blocks"] < sum(-(-t // 16) for t in st.seq_lens.tolist())


def test_long_small_tables_partition_pool():
    wl = workloads.long(num_seqs=3, seq_len=320, num_q_heads=8, num_kv_heads=2, head_dim=32)
    st = wl.steps[0]
    _check_step_invariants(wl, st)
    assert sorted(st.block_tables.flatten().tolist()) == list(range(wl.num_blocks))


def test_cb_small_steps():
    wl = workloads.cb(num_seqs=8, num_q_heads=4, num_kv_heads=2, head_dim=32, max_len0=70,
                      chunk=40, num_steps=3, num_blocks=512)
    prev = None
    for st in wl.steps:
        _check_step_invariants(wl, st)
        assert st.slot_mapping.numel() == 8 - 1 + 41
        if prev is not None:
            grew = (st.seq_lens - prev.seq_lens).tolist()
            assert sorted(grew) == [1] * 7 + [41]
            # tables only ever append
            for i in range(8):
                keep = -(-int(prev.seq_lens[i]) // 16)
                assert torch.equal(st.block_tables[i, :keep], prev.block_tables[i, :keep])
        prev = st


def test_full_size_shapes_are_as_specified():
    """Cheap structural facts of the full configurations (no cache fill)."""
    rng = np.random.default_rng(2)
    lens = rng.integers(128, 2049, size=32)
    assert lens.min() >= 128 and lens.max() <= 2048
    assert math.ceil(4096 + 10 * 2049) / 16 <= 1537


def test_fork_copy_on_write_and_swap():
    pool = BlockPool(10, 4)
    pool.add("A", 6)                                   # [0, 1], tail half full
    pool.fork("A", "B")
    assert pool.ref_cnt[:2] == [2, 2]
    with pytest.raises(SharedTailWrite):
        pool.grow("B", 1)
    assert pool.copy_on_write("B") == (1, 2)
    assert pool.tables["B"] == [0, 2] and pool.ref_cnt[:3] == [2, 1, 1]
    assert pool.copy_on_write("B") is None             # already private
    pool.grow("B", 3)                                  # fills block 2, takes block 3
    assert pool.tables["B"] == [0, 2, 3]
    # swap: private blocks only
    host = BlockPool(6, 4)
    with pytest.raises(SharedTailWrite):
        pool.swap_out("B", host)                       # block 0 shared with A
    pool.add("C", 9)                                   # [4, 5, 6]
    pairs = pool.swap_out("C", host)
    assert pairs == [(4, 0), (5, 1), (6, 2)] and "C" not in pool.tables
    assert list(pool.free_queue)[-3:] == [4, 5, 6] and host.lengths["C"] == 9
    back = pool.swap_in("C", host)
    assert [h for h, _ in back] == [0, 1, 2] and pool.lengths["C"] == 9
    assert host.num_free == 6
    # all-or-nothing on a full host pool
    small = BlockPool(2, 4)
    before = (list(pool.free_queue), dict(pool.tables))
    with pytest.raises(MemoryError):
        pool.swap_out("C", small)
    assert (list(pool.free_queue), dict(pool.tables)) == before


def test_append_step_follows_the_append_rule():
    """A decode step's appends: a full tail takes a fresh block, a shared
    partly filled tail is copied first (one copy for the first of its
    sharers; the last sharer then owns it alone), a private tail is written
    in place; all or nothing when the pool runs short."""
    pool = BlockPool(10, 4, free_order=range(10))
    pool.add("A", 6)                                   # [0, 1]: tail 1 half full
    pool.fork("A", "B")                                # shares 0 and 1
    pool.add("C", 8)                                   # [2, 3]: tail full
    pool.add("D", 2)                                   # [4]: private, half full
    pairs = pool.append_step(["A", "B", "C", "D"])
    assert pairs == [(1, 5)]                           # A copies the shared tail
    assert pool.tables["A"] == [0, 5] and pool.tables["B"] == [0, 1]
    assert pool.ref_cnt[1] == 1 and pool.ref_cnt[5] == 1
    assert pool.tables["C"] == [2, 3, 6] and pool.tables["D"] == [4]
    assert [pool.lengths[s] for s in "ABCD"] == [7, 7, 9, 3]
    # the new positions' slots are where pa_decode_append writes
    assert pool.slot("A", 6) == 5 * 4 + 2 and pool.slot("C", 8) == 6 * 4
    # all or nothing: one block left, a step that needs two changes nothing
    assert pool.num_free == 3
    pool.add("E", 4)                                   # block 7, full
    pool.add("F", 4)                                   # block 8, full
    before = (list(pool.free_queue), {k: list(v) for k, v in pool.tables.items()},
              dict(pool.lengths), list(pool.ref_cnt))
    with pytest.raises(MemoryError):
        pool.append_step(["A", "E", "F"])              # A in place, E and F a block each
    assert (list(pool.free_queue), {k: list(v) for k, v in pool.tables.items()},
            dict(pool.lengths), list(pool.ref_cnt)) == before
    assert pool.append_step(["A", "E"]) == [] and pool.tables["E"] == [7, 9]
    with pytest.raises(ValueError):
        pool.append_step(["A", "A"])


def test_positions_give_the_slot_mapping():
    """Every workload's (seq_id, position) per new token maps, through the
    oracle's addressing, to the slot mapping the host pool produced."""
    for wl in (workloads.tiny(),
               workloads.mha(num_seqs=6, num_heads=4, head_dim=32, min_len=20, max_len=90,
                             num_blocks=64),
               workloads.cb(num_seqs=8, num_q_heads=4, num_kv_heads=2, head_dim=32,
                            max_len0=70, chunk=40, num_steps=3, num_blocks=512)):
        for st in wl.steps:
            got = oracle.slots_from_positions(st.seq_ids, st.positions, st.block_tables,
                                              wl.block_size)
            assert got.tolist() == st.slot_mapping.tolist()


def test_shared_prefix_groups_from_the_pool():
    """Sequences sharing leading blocks (ref_cnt > 1) group by their first
    block; the shared count is the run of entries every member agrees on;
    singletons and unshared sequences are left out."""
    pool = BlockPool(64, 4)
    pool.add("a", 10)                               # 3 blocks
    pool.add("b", 14, prefix_of="a", prefix_tokens=8)
    pool.add("c", 9, prefix_of="a", prefix_tokens=4)
    pool.add("d", 5)
    pool.fork("d", "e")
    pool.add("f", 3)
    seqs = ["f", "a", "b", "c", "d", "e"]
    groups = sorted(pool.shared_prefix_groups(seqs))
    # a, b, c share block 0 (c only that one); d and e share all of d's blocks
    assert groups == [([1, 2, 3], 1), ([4, 5], 2)]
    assert pool.shared_prefix_groups(["f", "a"]) == []


def test_prefix_groups_marshal_to_csr():
    grp = pa.prefix_groups([([4, 1], 3), ([7], 9), ([0, 2, 5], 2)], 8)
    assert grp.num_groups == 2                      # the one-member group is dropped
    assert grp.seq_group.tolist() == [1, 0, 1, -1, 0, 1, -1, -1]
    assert grp.member_start.tolist() == [0, 2, 5]
    assert grp.members.tolist() == [4, 1, 0, 2, 5]
    assert grp.prefix_blocks.tolist() == [3, 2]
    assert (grp.max_group_size, grp.max_prefix_blocks) == (3, 3)
    assert all(t.dtype == torch.int32 for t in (grp.seq_group, grp.member_start,
                                                grp.members, grp.prefix_blocks))
    empty = pa.prefix_groups([], 3)
    assert empty.num_groups == 0 and empty.seq_group.tolist() == [-1, -1, -1]
