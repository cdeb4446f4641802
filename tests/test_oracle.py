"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check is a plain function so that the mutation test at the bottom can
run the whole set against deliberately broken builds of the oracle: each
plausible mistake (wrong GQA mapping, dropped scale, off-by-one offset,
K and V swapped, missing normalisation, transposed cache index, wrong merge
sign, ...) must make at least one check fail.
"""
import itertools
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_109_gb300 import workloads
from tests.conftest import golden

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


# ---- helpers that build inputs the way the pages do ------------------------

def place_blocks(contiguous, tables, lengths, num_blocks, block_size):
    """Paged cache built the glossary script's way: for each table entry, copy
    that logical block's contiguous segment into the physical block.
    contiguous[s] is [Hkv, T_s, D]."""
    hkv, _, d = contiguous[0].shape
    cache = torch.zeros(num_blocks, hkv, block_size, d, dtype=contiguous[0].dtype)
    for s, table in enumerate(tables):
        for logical, physical in enumerate(table):
            if physical < 0:
                continue
            start = logical * block_size
            end = min(start + block_size, lengths[s])
            if start < end:
                cache[physical, :, : end - start] = contiguous[s][:, start:end]
    return cache


def random_case(gen, n, hq, hkv, d, bs, lengths, num_blocks, dtype=torch.float32):
    """Contiguous K/V per sequence, random injective tables, paged caches."""
    contiguous_k = [torch.randn(hkv, t, d, generator=gen).to(dtype) for t in lengths]
    contiguous_v = [torch.randn(hkv, t, d, generator=gen).to(dtype) for t in lengths]
    need = [-(-t // bs) for t in lengths]
    perm = torch.randperm(num_blocks, generator=gen).tolist()
    width = max(max(need), 1)
    tables, pos = [], 0
    for k in need:
        tables.append(perm[pos: pos + k] + [-1] * (width - k))
        pos += k
    kc = place_blocks(contiguous_k, tables, lengths, num_blocks, bs)
    vc = place_blocks(contiguous_v, tables, lengths, num_blocks, bs)
    q = torch.randn(n, hq, d, generator=gen).to(dtype)
    return (q, kc, vc, torch.tensor(tables, dtype=torch.int32),
            torch.tensor(lengths, dtype=torch.int32), contiguous_k, contiguous_v)


def expand_kv(x, hq):
    """Query-head view of kv rows, grouped as the glossary script does."""
    return x.repeat_interleave(hq // x.shape[0], dim=0)


# ---- checks -----------------------------------------------------------------

def check_addressing():
    for case in golden("addressing.json")["cases"]:
        for p, s in zip(case["positions"], case["slots"]):
            got = oracle.physical_slot(case["table"], case["block_size"], p)
            assert got == s, (case["cite"], p, got, s)
    assert oracle.physical_slot([5, 3, -1], 4, 9) == -1   # padding entry


def check_block_counts():
    g = golden("block_counts.json")
    bs = g["block_size"]
    blocks = [oracle.blocks_needed(n, bs) for n in g["lengths"]]
    assert blocks == g["blocks"]
    assert sum(blocks) == g["total_blocks"] > g["pool_blocks"]
    assert [oracle.tail_waste(n, bs) for n in g["lengths"]] == g["tail_waste"]
    assert all(0 <= oracle.tail_waste(n, bs) < bs for n in range(1, 100))
    assert len(g["lengths"]) * g["reserve_max_len"] == g["reserved_slots"]
    assert sum(g["lengths"]) == g["live_tokens"]


def check_worked_example_write():
    """The 13 writes of the worked example rebuild the script's physical cache."""
    g = golden("shared_prefix.json")
    wl = workloads.tiny()
    st = wl.steps[0]
    ref_k = place_blocks(wl.contiguous_k, g["tables"], g["lengths"], g["num_blocks"],
                         g["block_size"])
    ref_v = place_blocks(wl.contiguous_v, g["tables"], g["lengths"], g["num_blocks"],
                         g["block_size"])
    kc = torch.zeros_like(ref_k)
    vc = torch.zeros_like(ref_v)
    slots = torch.tensor(g["derived_slot_mapping"]["slots"], dtype=torch.int64)
    assert oracle.write_kv(st.k_new, st.v_new, slots, kc, vc) == 0
    assert torch.equal(kc, ref_k) and torch.equal(vc, ref_v)
    # physical blocks 0, 2 and 4 are never referenced and stay zero
    assert not kc[[0, 2, 4]].any()


def check_worked_example_paged_equals_contiguous():
    """Script check: paged attention equals dense attention on contiguous
    K/V, max abs difference printed as exactly 0."""
    g = golden("shared_prefix.json")
    wl = workloads.tiny()
    st = wl.steps[0]
    kc = place_blocks(wl.contiguous_k, g["tables"], g["lengths"], 7, 4)
    vc = place_blocks(wl.contiguous_v, g["tables"], g["lengths"], 7, 4)
    out = oracle.decode(st.q, kc, vc, st.block_tables, st.seq_lens, wl.scale)
    max_diff = 0.0
    for s in range(2):
        ek = expand_kv(wl.contiguous_k[s], 4)
        ev = expand_kv(wl.contiguous_v[s], 4)
        for h in range(4):
            dense = oracle.attend(st.q[s, h].numpy(), ek[h].numpy(), ev[h].numpy(), wl.scale)
            max_diff = max(max_diff, float(np.abs(out[s, h] - dense).max()))
    assert max_diff == g["max_attention_abs_diff"]


def check_sdpa_special_case():
    """Library special case: torch SDPA in fp64 on the contiguous K/V with
    repeat_interleave'd heads."""
    gen = torch.Generator().manual_seed(7)
    for (hq, hkv, d, bs, lengths) in [(4, 2, 8, 4, (10, 7)), (8, 2, 16, 2, (1, 5, 33)),
                                      (6, 3, 32, 8, (17, 64, 3, 40))]:
        q, kc, vc, bt, sl, ck, cv = random_case(gen, len(lengths), hq, hkv, d, bs, lengths,
                                                 64)
        scale = 1.0 / math.sqrt(d) * 1.3
        out = oracle.decode(q, kc, vc, bt, sl, scale)
        for s, t in enumerate(lengths):
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[s].double()[:, None, :], expand_kv(ck[s].double(), hq),
                expand_kv(cv[s].double(), hq), scale=scale)[:, 0, :]
            assert np.abs(out[s] - ref.numpy()).max() < 1e-12


def check_gqa_grouping():
    """Head h of a group reads kv head h // (Hq/Hkv): constant V per kv head."""
    hq, hkv, d, bs, t = 6, 3, 4, 4, 9
    kc = torch.randn(4, hkv, bs, d, generator=torch.Generator().manual_seed(1))
    vc = torch.zeros(4, hkv, bs, d)
    for g in range(hkv):
        vc[:, g] = float(g + 1)
    q = torch.randn(1, hq, d, generator=torch.Generator().manual_seed(2))
    out = oracle.decode(q, kc, vc, torch.tensor([[2, 0, 3]], dtype=torch.int32),
                        torch.tensor([t], dtype=torch.int32), 0.5)
    owner = torch.arange(hkv).repeat_interleave(hq // hkv)
    for h in range(hq):
        assert np.allclose(out[0, h], float(owner[h] + 1), rtol=0, atol=1e-14)


def check_closed_forms():
    gen = torch.Generator().manual_seed(11)
    hq, hkv, d, bs = 4, 2, 8, 4
    lengths = (9, 1, 6)
    q, kc, vc, bt, sl, ck, cv = random_case(gen, 3, hq, hkv, d, bs, lengths, 16)
    # q = 0: uniform weights, out = mean of the visible V rows
    out = oracle.decode(torch.zeros_like(q), kc, vc, bt, sl, 0.35)
    for s, t in enumerate(lengths):
        ev = expand_kv(cv[s].double(), hq)
        assert np.abs(out[s] - ev.mean(dim=1).numpy()).max() < 1e-14
    # T = 1: out = v_0 exactly
    out = oracle.decode(q, kc, vc, bt, sl, 0.35)
    assert np.array_equal(out[1], expand_kv(cv[1].double(), hq)[:, 0].numpy())
    # constant V rows: out = that constant
    vconst = torch.full_like(vc, -1.25)
    out = oracle.decode(q, kc, vconst, bt, sl, 0.35)
    assert np.abs(out + 1.25).max() < 1e-14
    # one dominant key (score gap > 50): out = its V row
    kdom = kc.clone()
    j = 4                                       # sequence 0, position 4
    blk = int(bt[0, j // bs])
    kdom[blk, 0, j % bs] = q[0, 0] * 80.0
    out = oracle.decode(q, kdom, vc, bt, sl, 1.0)
    assert np.abs(out[0, 0] - cv[0][0, j].double().numpy()).max() < 1e-12
    # two tokens, hand-computed weights: w1 = 1 / (1 + exp(-(s1 - s0)))
    q2 = torch.tensor([[[1.0, 2.0]]])
    k2 = torch.tensor([[[[0.5, 0.0], [0.0, 1.0]]]])     # [1 block, 1 head, 2, 2]
    v2 = torch.tensor([[[[3.0, -1.0], [7.0, 5.0]]]])
    out = oracle.decode(q2, k2, v2, torch.tensor([[0]], dtype=torch.int32),
                        torch.tensor([2], dtype=torch.int32), 0.7)
    s0, s1 = 0.7 * 0.5, 0.7 * 2.0
    w1 = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    expect = np.array([3.0 * (1 - w1) + 7.0 * w1, -1.0 * (1 - w1) + 5.0 * w1])
    assert np.abs(out[0, 0] - expect).max() < 1e-14


def check_relabel_invariance():
    """Permuting physical block ids together with the tables changes nothing."""
    gen = torch.Generator().manual_seed(12)
    q, kc, vc, bt, sl, _, _ = random_case(gen, 3, 4, 2, 8, 4, (13, 4, 7), 12)
    out = oracle.decode(q, kc, vc, bt, sl, 0.4)
    perm = torch.randperm(12, generator=gen)
    kp = torch.empty_like(kc)
    vp = torch.empty_like(vc)
    kp[perm] = kc
    vp[perm] = vc
    btp = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    assert np.array_equal(oracle.decode(q, kp, vp, btp, sl, 0.4), out)


def check_brute_force_tables():
    """Every injective table over a pool of n+1 blocks, B in {1, 2, 4}: paged
    decode equals dense attention on the contiguous rows, exactly."""
    gen = torch.Generator().manual_seed(13)
    hq, hkv, d = 2, 1, 4
    cases = 0
    for bs, tmax in ((1, 4), (2, 8), (4, 8)):
        for t in range(1, tmax + 1):
            n = -(-t // bs)
            ck = torch.randn(hkv, t, d, generator=gen)
            cv = torch.randn(hkv, t, d, generator=gen)
            q = torch.randn(1, hq, d, generator=gen)
            dense = [oracle.attend(q[0, h].numpy(), expand_kv(ck, hq)[h].numpy(),
                                   expand_kv(cv, hq)[h].numpy(), 0.6) for h in range(hq)]
            for table in itertools.permutations(range(n + 1), n):
                kc = place_blocks([ck], [list(table)], [t], n + 1, bs)
                vc = place_blocks([cv], [list(table)], [t], n + 1, bs)
                out = oracle.decode(q, kc, vc, torch.tensor([table], dtype=torch.int32),
                                    torch.tensor([t], dtype=torch.int32), 0.6)
                for h in range(hq):
                    assert np.array_equal(out[0, h], dense[h]), (bs, t, table)
                cases += 1
    assert cases > 100


def check_partition_merge():
    """Blockwise rewrite: per-partition (m, l, acc) merged by log-sum-exp
    equals the single softmax over all tokens (paper notes, 10-token example,
    partitions = blocks of 4)."""
    gen = torch.Generator().manual_seed(14)
    lengths = (10, 1, 37, 100)
    q, kc, vc, bt, sl, ck, cv = random_case(gen, 4, 4, 2, 8, 4, lengths, 64)
    full = oracle.decode(q, kc, vc, bt, sl, 0.3)
    for part in (1, 3, 4, 16, 100, 105):
        m, l, acc = oracle.decode_partials(q, kc, vc, bt, sl, 0.3, part)
        for s, t in enumerate(lengths):
            n = -(-t // part)
            assert np.isnan(m[s, :, n:]).all()
            for h in range(4):
                merged = oracle.merge(m[s, h, :n], l[s, h, :n], acc[s, h, :n])
                assert np.abs(merged - full[s, h]).max() < 1e-13, (part, s, h)
    # single partition: m is the max score, acc / l is the output
    m, l, acc = oracle.decode_partials(q, kc, vc, bt, sl, 0.3, 1000)
    for s, t in enumerate(lengths):
        for h in range(4):
            scores = 0.3 * (expand_kv(ck[s].double(), 4)[h] @ q[s, h].double())
            assert abs(m[s, h, 0] - float(scores.max())) < 1e-14
            assert abs(l[s, h, 0] - float(torch.exp(scores - scores.max()).sum())) < 1e-12
            assert np.abs(acc[s, h, 0] / l[s, h, 0] - full[s, h]).max() < 1e-13


def check_write_semantics():
    gen = torch.Generator().manual_seed(15)
    nb, hkv, bs, d = 5, 3, 4, 8
    k = torch.randn(6, hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(6, hkv, d, generator=gen).to(torch.bfloat16)
    kc = torch.zeros(nb, hkv, bs, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    slots = torch.tensor([3, -1, 17, 20, 0, 19], dtype=torch.int64)   # 20 == nb*bs: rejected
    assert oracle.write_kv(k, v, slots, kc, vc) == 1
    written = {3: 0, 17: 2, 0: 4, 19: 5}
    for s in range(nb * bs):
        blk, row = divmod(s, bs)
        if s in written:
            assert torch.equal(kc[blk, :, row], k[written[s]])
            assert torch.equal(vc[blk, :, row], v[written[s]])
        else:
            assert not kc[blk, :, row].any() and not vc[blk, :, row].any()
    # a later token wins when two write one slot (sequential order)
    slots2 = torch.tensor([7, 7], dtype=torch.int64)
    oracle.write_kv(k[:2], v[:2], slots2, kc, vc)
    assert torch.equal(kc[1, :, 3], k[1])


def check_write_then_read_roundtrip():
    """Tokens scattered through a table's slots read back as the dense rows."""
    gen = torch.Generator().manual_seed(16)
    hq, hkv, d, bs, t = 4, 2, 8, 4, 11
    table = [6, 2, 9]
    ck = torch.randn(t, hkv, d, generator=gen)
    cv = torch.randn(t, hkv, d, generator=gen)
    slots = torch.tensor([table[p // bs] * bs + p % bs for p in range(t)], dtype=torch.int64)
    kc = torch.zeros(10, hkv, bs, d)
    vc = torch.zeros(10, hkv, bs, d)
    oracle.write_kv(ck, cv, slots, kc, vc)
    q = torch.randn(1, hq, d, generator=gen)
    out = oracle.decode(q, kc, vc, torch.tensor([table], dtype=torch.int32),
                        torch.tensor([t], dtype=torch.int32), 0.5)
    ek = expand_kv(ck.permute(1, 0, 2), hq)
    ev = expand_kv(cv.permute(1, 0, 2), hq)
    for h in range(hq):
        assert np.array_equal(out[0, h], oracle.attend(q[0, h].numpy(), ek[h].numpy(),
                                                       ev[h].numpy(), 0.5))


def check_bf16_widening():
    """bf16 inputs are widened exactly (values representable in bf16)."""
    vals = torch.tensor([1.0, -2.5, 0.15625, 3.0e38, -1.0e-38, 0.0])
    b = vals.to(torch.bfloat16)
    kc = torch.zeros(1, 1, 6, 1, dtype=torch.bfloat16)
    kc[0, 0, :, 0] = b
    # q = 0 -> mean of V; V = K here; compare against float64 mean of the same bits
    out = oracle.decode(torch.zeros(1, 1, 1, dtype=torch.bfloat16), kc, kc,
                        torch.tensor([[0]], dtype=torch.int32),
                        torch.tensor([1], dtype=torch.int32), 1.0)
    assert out[0, 0, 0] == float(b[0].double())


def check_zero_length():
    """T = 0 yields a zero output row (reading: no visible token, no weight)."""
    kc = torch.randn(2, 1, 4, 8)
    out = oracle.decode(torch.randn(2, 2, 8), kc, kc, torch.tensor([[0], [1]], dtype=torch.int32),
                        torch.tensor([0, 3], dtype=torch.int32), 0.5)
    assert not out[0].any() and np.isfinite(out[1]).all()


def check_copy_blocks():
    """Whole-block copies, in pair order; out-of-range pairs are skipped."""
    gen = torch.Generator().manual_seed(17)
    src_k = torch.randn(6, 2, 4, 8, generator=gen).to(torch.bfloat16)
    src_v = torch.randn(6, 2, 4, 8, generator=gen).to(torch.bfloat16)
    dst_k = torch.zeros(3, 2, 4, 8, dtype=torch.bfloat16)
    dst_v = torch.zeros_like(dst_k)
    pairs = [[4, 0], [1, 2], [7, 1], [0, 3], [2, -1]]
    assert oracle.copy_blocks(src_k, src_v, dst_k, dst_v, pairs) == 3
    assert torch.equal(dst_k[0], src_k[4]) and torch.equal(dst_v[0], src_v[4])
    assert torch.equal(dst_k[2], src_k[1]) and torch.equal(dst_v[2], src_v[1])
    assert not dst_k[1].any() and not dst_v[1].any()
    # inside one pool, in order: block 5 <- 0, then block 3 <- 5 (now block 0's data)
    k, v = src_k.clone(), src_v.clone()
    assert oracle.copy_blocks(k, v, k, v, [[0, 5], [5, 3]]) == 0
    assert torch.equal(k[3], src_k[0]) and torch.equal(v[5], src_v[0])
    assert torch.equal(k[1], src_k[1])


def check_slots_from_positions():
    """Slots from (sequence, position) agree with the pages' addressing values."""
    cases = golden("addressing.json")["cases"]
    for case in cases:
        bs = case["block_size"]
        width = max(len(c["table"]) for c in cases if c["block_size"] == bs)
        tables = [c["table"] + [-1] * (width - len(c["table"]))
                  for c in cases if c["block_size"] == bs]
        row = tables.index(case["table"] + [-1] * (width - len(case["table"])))
        n = len(case["positions"])
        got = oracle.slots_from_positions([row] * n, case["positions"], tables, bs)
        assert got.tolist() == case["slots"], case["cite"]
    got = oracle.slots_from_positions([0, -1, 0, 2, 0], [1, 3, -2, 0, 12],
                                      [[7, 3, 11], [1, 2, 3]], 4)
    assert got.tolist() == [29, -1, -1, -1, -1]   # skip, skip, bad seq, past the table


def check_copy_on_write_scenario():
    """nxmr.cn article §4.2: two branches share a partly filled last block;
    the writing branch first copies it into a fresh block and re-points its
    table; the other branch's data and output are unchanged."""
    from paged_kv_cache_109_gb300.block_pool import BlockPool
    gen = torch.Generator().manual_seed(18)
    hq, hkv, d, bs = 4, 2, 8, 4
    pool = BlockPool(8, bs, free_order=[6, 2, 5, 0, 1, 3, 4, 7])
    pool.add("A", 6)                        # blocks [6, 2], last one half full
    pool.fork("A", "B")                     # B shares both
    kc = torch.randn(8, hkv, bs, d, generator=gen)
    vc = torch.randn(8, hkv, bs, d, generator=gen)
    q = torch.randn(2, hq, d, generator=gen)
    before = oracle.decode(q[:1], kc, vc, torch.tensor([pool.tables["A"]], dtype=torch.int32),
                           torch.tensor([6], dtype=torch.int32), 0.5)
    pair = pool.copy_on_write("B")
    assert pair == (2, 5) and pool.tables["B"] == [6, 5] and pool.ref_cnt[2] == 1
    assert oracle.copy_blocks(kc, vc, kc, vc, [pair]) == 0
    pool.grow("B", 1)
    new_k = torch.randn(1, hkv, d, generator=gen)
    new_v = torch.randn(1, hkv, d, generator=gen)
    slot = pool.slot("B", 6)
    assert slot == 5 * bs + 2
    oracle.write_kv(new_k, new_v, torch.tensor([slot]), kc, vc)
    tables = torch.tensor([pool.tables["A"], pool.tables["B"]], dtype=torch.int32)
    out = oracle.decode(q, kc, vc, tables, torch.tensor([6, 7], dtype=torch.int32), 0.5)
    assert np.array_equal(out[0], before[0])            # A untouched
    # B = dense attention over A's 6 rows plus its own new row
    rows_k = torch.cat([kc[6], kc[2, :, :2], new_k.permute(1, 0, 2)], 1)   # [Hkv, 7, D]
    rows_v = torch.cat([vc[6], vc[2, :, :2], new_v.permute(1, 0, 2)], 1)
    for h in range(hq):
        ref = oracle.attend(q[1, h].numpy(), expand_kv(rows_k, hq)[h].numpy(),
                            expand_kv(rows_v, hq)[h].numpy(), 0.5)
        assert np.abs(out[1, h] - ref).max() < 1e-14


def check_prefill_causal_sdpa():
    """Multi-query rows are the last L_i positions of T_i and see keys up to
    their own position: torch SDPA (fp64) with an explicit bottom-right
    causal mask on the contiguous K/V is the library special case."""
    gen = torch.Generator().manual_seed(19)
    hq, hkv, d, bs = 8, 2, 16, 4
    lengths = (9, 21, 1, 40)
    qlens = (9, 5, 1, 17)              # a whole prompt, a chunk, a decode row, a chunk
    _, kc, vc, bt, sl, ck, cv = random_case(gen, 4, hq, hkv, d, bs, lengths, 64)
    qs = [0]
    for L in qlens:
        qs.append(qs[-1] + L)
    q = torch.randn(qs[-1], hq, d, generator=gen)
    out = oracle.prefill(q, qs, kc, vc, bt, sl, 0.3)
    for i, (T, L) in enumerate(zip(lengths, qlens)):
        rows = q[qs[i]:qs[i + 1]].double().permute(1, 0, 2)            # [Hq, L, D]
        pos = torch.arange(T - L, T)
        mask = torch.arange(T)[None, :] <= pos[:, None]                # [L, T]
        ref = torch.nn.functional.scaled_dot_product_attention(
            rows, expand_kv(ck[i].double(), hq), expand_kv(cv[i].double(), hq),
            attn_mask=mask, scale=0.3).permute(1, 0, 2)
        assert np.abs(out[qs[i]:qs[i + 1]] - ref.numpy()).max() < 1e-12


def check_prefill_last_row_is_decode():
    """The last query row of every sequence is the single-query decode."""
    gen = torch.Generator().manual_seed(20)
    _, kc, vc, bt, sl, _, _ = random_case(gen, 3, 4, 2, 8, 4, (13, 6, 30), 32)
    qs = [0, 4, 5, 12]
    q = torch.randn(12, 4, 8, generator=gen)
    out = oracle.prefill(q, qs, kc, vc, bt, sl, 0.4)
    last = [qs[i + 1] - 1 for i in range(3)]
    dec = oracle.decode(q[last], kc, vc, bt, sl, 0.4)
    assert np.array_equal(out[last], dec)


CHECKS = [check_addressing, check_block_counts, check_worked_example_write,
          check_worked_example_paged_equals_contiguous, check_sdpa_special_case,
          check_gqa_grouping, check_closed_forms, check_relabel_invariance,
          check_brute_force_tables, check_partition_merge, check_write_semantics,
          check_write_then_read_roundtrip, check_bf16_widening, check_zero_length,
          check_copy_blocks, check_slots_from_positions, check_copy_on_write_scenario,
          check_prefill_causal_sdpa, check_prefill_last_row_is_decode]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check()


# ---- mutation test: the pins must reject plausible oracle mistakes ----------

MUTANTS = [
    ("gqa head mapping", "(int32_t)(h / group)", "(int32_t)(h % num_kv_heads)"),
    ("offset off by one", "int64_t offset = position % block_size;",
     "int64_t offset = (position + 1) % block_size;"),
    ("table lookup skipped", "int64_t physical = table[logical];",
     "int64_t physical = table[logical] * 0 + logical;"),
    ("scale dropped", "s[t] = scale * dot;", "s[t] = dot;"),
    ("V gathered from K", "gather_rows(v_cache", "gather_rows(k_cache"),
    ("normalisation dropped", "out[d] /= l;", "out[d] /= 1.0;"),
    ("head and row transposed",
     "((block * num_kv_heads + g) * block_size + row) * head_dim",
     "((block * num_kv_heads + row % num_kv_heads) * block_size + g % block_size) * head_dim"),
    ("merge weight sign", "double w = exp(m[p] - M);", "double w = exp(M - m[p]);"),
    ("partial weight unscaled", "double w = exp(scale * dot - m);", "double w = exp(dot - m);"),
    ("write row off by one", "int64_t row = s % block_size;",
     "int64_t row = (s + 1) % block_size;"),
    ("query head of group", "(i * num_q_heads + h) * head_dim + d",
     "(i * num_q_heads + h / group * group) * head_dim + d"),
    ("partition max missing", "if (scale * dot > m) m = scale * dot;", "m = 0.0;"),
    ("block copy V from K", "(const char*)src_v + s * block_bytes", "(const char*)src_k + s * block_bytes"),
    ("slots from the first table", "oracle_slot(block_tables + s * max_blocks,",
     "oracle_slot(block_tables + 0 * max_blocks,"),
    ("causal mask drops the diagonal", "int64_t n = p + 1;", "int64_t n = p;"),
    ("no causal mask", "int64_t n = p + 1;", "int64_t n = T;"),
    ("query position off by one", "int64_t p = T - L + (r - query_start[i]);",
     "int64_t p = T - L + (r - query_start[i]) - 1;"),
]


@pytest.mark.parametrize("name,before,after", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, before, after):
    src = open(oracle._SRC).read()
    assert before in src, f"mutation target not found: {before}"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(before, after))
    lib = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", lib, str(mutant), "-lm"],
                   check=True, capture_output=True)
    failed = []
    with oracle.using(lib):
        for check in CHECKS:
            try:
                check()
            except (AssertionError, ValueError):
                failed.append(check.__name__)
    assert failed, f"mutant '{name}' passed every pin"
