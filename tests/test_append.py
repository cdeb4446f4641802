"""pa_decode_append (one decode step in one call: each sequence's newest token
written at position seq_lens - 1, then the decode) on the GPU.  Its caches
must equal the oracle's write bit for bit, its output the oracle's decode
within the stated bound, and both must equal pa_write_kv_positions followed by
pa_decode bit for bit, on the fused TMA path and on every fallback kernel."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import workloads
from paged_kv_cache_109_gb300.block_pool import BlockPool
from tests._gpu import (BF16_ATOL, BF16_RTOL, DeviceState, HostState, assert_close,
                        sample_pairs, tolerance)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clear_device_error(cuda_device):
    pa.last_device_error()
    yield


def _batch(hkv, group, d, bs, dtype, lens, seed, spare=3):
    """Caches, private tables (no block shared), q and the new rows; the
    appended slots of the caches hold NaN, which no output may show."""
    g = torch.Generator().manual_seed(seed)
    need = [max(1, -(-t // bs)) for t in lens]
    nb = sum(need) + spare
    perm = torch.randperm(nb, generator=g).tolist()
    width, pos, rows = max(need) + 1, 0, []
    for k in need:
        rows.append(perm[pos:pos + k] + [-1] * (width - k))
        pos += k
    bt = torch.tensor(rows, dtype=torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    for i, t in enumerate(lens):
        if t > 0:
            blk = int(bt[i, (t - 1) // bs])
            kc[blk, :, (t - 1) % bs] = float("nan")
            vc[blk, :, (t - 1) % bs] = float("nan")
    n = len(lens)
    q = torch.randn(n, hkv * group, d, generator=g).to(dtype)
    k_new = torch.randn(n, hkv, d, generator=g).to(dtype)
    v_new = torch.randn(n, hkv, d, generator=g).to(dtype)
    return kc, vc, bt, sl, q, k_new, v_new


def _run_both(dev, kc, vc, bt, sl, q, k_new, v_new, max_len, part, scale):
    """(fused call's out and caches, write-then-decode out and caches)."""
    bt_d, sl_d = bt.to(dev), sl.to(dev)
    kd, vd = kc.to(dev), vc.to(dev)
    out = pa.decode_append(q.to(dev), k_new.to(dev), v_new.to(dev), kd, vd, bt_d, sl_d, max_len,
                           scale, partition_tokens=part)
    kr, vr = kc.to(dev), vc.to(dev)
    n = sl.numel()
    pa.write_kv_positions(k_new.to(dev), v_new.to(dev),
                          torch.arange(n, dtype=torch.int32, device=dev), (sl - 1).to(dev),
                          bt_d, kr, vr)
    ref = pa.decode(q.to(dev), kr, vr, bt_d, sl_d, max_len, scale, partition_tokens=part)
    torch.cuda.synchronize()
    return (out.cpu(), kd.cpu(), vd.cpu()), (ref.cpu(), kr.cpu(), vr.cpu())


def _oracle(kc, vc, bt, sl, q, k_new, v_new, bs, scale):
    n = sl.numel()
    slots = torch.from_numpy(oracle.slots_from_positions(
        torch.arange(n, dtype=torch.int32), sl - 1, bt, bs))
    kh, vh = kc.clone(), vc.clone()
    assert oracle.write_kv(k_new, v_new, slots, kh, vh) == 0
    return oracle.decode(q, kh, vh, bt, sl, scale), kh, vh


# (kv heads, group, head dim, block size, dtype, partition): the TMA kernel
# (fused) for the first eight, then the mma.sync, tiled and generic kernels
# (cache write first)
SHAPES = [
    (8, 4, 128, 16, torch.bfloat16, 0),
    (8, 4, 128, 16, torch.bfloat16, 64),
    (2, 16, 64, 8, torch.bfloat16, 32),
    (4, 1, 96, 32, torch.bfloat16, 64),
    (2, 32, 112, 16, torch.bfloat16, 64),      # two sub-groups per kv head
    (4, 8, 80, 64, torch.bfloat16, 128),
    (1, 5, 128, 256, torch.bfloat16, 256),
    (2, 4, 32, 16, torch.bfloat16, 64),        # head dim 32: one box, half zero-filled
    (2, 8, 48, 24, torch.bfloat16, 48),        # mma.sync kernel
    (2, 2, 96, 4, torch.bfloat16, 32),         # tiled kernel, bf16
    (2, 4, 128, 16, torch.float32, 64),        # tiled kernel, fp32
    (2, 3, 20, 5, torch.bfloat16, 20),         # generic kernel
    (2, 4, 256, 16, torch.bfloat16, 64),       # TMA kernel at head dim 256, write first
]


@pytest.mark.parametrize("hkv,group,d,bs,dtype,part", SHAPES)
def test_append_matches_write_then_decode_and_oracle(cuda_device, hkv, group, d, bs, dtype,
                                                     part):
    p = part or 1024
    lens = [0, 1, bs - 1, bs, bs + 1, p, p + 1, 2 * p + bs, 3 * p - 1, 777, 5]
    lens = [t for t in lens if t >= 0]
    kc, vc, bt, sl, q, k_new, v_new = _batch(hkv, group, d, bs, dtype, lens, seed=hkv * d + bs)
    max_len = int(sl.max())
    scale = 1 / math.sqrt(d)
    fused = SHAPES.index((hkv, group, d, bs, dtype, part)) < 8
    assert (pa.decode_path(hkv * group, kc) == 1) == (fused or d == 256)
    (out, kd, vd), (ref, kr, vr) = _run_both(cuda_device, kc, vc, bt, sl, q, k_new, v_new,
                                             max_len, part, scale)
    assert pa.last_device_error() == 0
    # one call equals the two, bit for bit
    assert torch.equal(kd.view(torch.uint8), kr.view(torch.uint8))
    assert torch.equal(vd.view(torch.uint8), vr.view(torch.uint8))
    assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
    # and the oracle: caches bit-exact, output within the bound
    oref, kh, vh = _oracle(kc, vc, bt, sl, q, k_new, v_new, bs, scale)
    assert torch.equal(kd.view(torch.uint8), kh.view(torch.uint8))
    assert torch.equal(vd.view(torch.uint8), vh.view(torch.uint8))
    atol, rtol = tolerance(dtype)
    assert_close(out.double().numpy(), oref, atol, rtol, f"append D={d} B={bs} G={group}")
    assert torch.isfinite(out.float()).all()


def test_unaligned_new_rows_take_the_separate_write(cuda_device):
    """k_new / v_new 2 bytes off a 16-byte boundary on a TMA shape: the write
    runs as its own kernel, with the same result."""
    hkv, group, d, bs = 8, 4, 128, 16
    lens = [300, 17, 1, 64]
    kc, vc, bt, sl, q, k_new, v_new = _batch(hkv, group, d, bs, torch.bfloat16, lens, seed=5)
    n = len(lens)
    dev = cuda_device
    flat_k = torch.empty(k_new.numel() + 1, dtype=torch.bfloat16, device=dev)
    flat_v = torch.empty(v_new.numel() + 1, dtype=torch.bfloat16, device=dev)
    kn = flat_k[1:].view(n, hkv, d)
    vn = flat_v[1:].view(n, hkv, d)
    kn.copy_(k_new.to(dev))
    vn.copy_(v_new.to(dev))
    kd, vd = kc.to(dev), vc.to(dev)
    out = pa.decode_append(q.to(dev), kn, vn, kd, vd, bt.to(dev), sl.to(dev), 300,
                           partition_tokens=64)
    torch.cuda.synchronize()
    oref, kh, vh = _oracle(kc, vc, bt, sl, q, k_new, v_new, bs, 1 / math.sqrt(d))
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    assert_close(out.cpu().double().numpy(), oref, BF16_ATOL, BF16_RTOL, "unaligned rows")
    assert pa.last_device_error() == 0


def test_pinned_host_new_rows(cuda_device):
    """q, k_new, v_new, tables and lengths in page-locked host memory: the
    kernels read them over the host link; same bits as device tensors."""
    hkv, group, d, bs = 8, 8, 128, 16
    lens = [1000, 33, 2049, 1]
    kc, vc, bt, sl, q, k_new, v_new = _batch(hkv, group, d, bs, torch.bfloat16, lens, seed=6)
    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    ref = pa.decode_append(q.to(dev), k_new.to(dev), v_new.to(dev), kd, vd, bt.to(dev),
                           sl.to(dev), 2049)
    kp, vp = kc.to(dev), vc.to(dev)
    out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    pa.decode_append(q.pin_memory(), k_new.pin_memory(), v_new.pin_memory(), kp, vp,
                     bt.pin_memory(), sl.pin_memory(), 2049, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), ref.cpu().view(torch.uint8))
    assert torch.equal(kp, kd) and torch.equal(vp, vd)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("d,bs", [(128, 16), (96, 4)])
def test_bad_length_or_table_entry_appends_nothing(cuda_device, d, bs):
    """A length past the host bound, and a bad table entry at the appended
    position, are reported; those sequences write nothing, the others are
    exact."""
    hkv, group = 2, 4
    lens = [100, 40, 70, 9]
    kc, vc, bt, sl, q, k_new, v_new = _batch(hkv, group, d, bs, torch.bfloat16, lens, seed=9)
    max_len = 100
    sl_bad = sl.clone()
    sl_bad[1] = max_len + 1                    # past the host bound (inside the table)
    bt_bad = bt.clone()
    bt_bad[2, (lens[2] - 1) // bs] = kc.shape[0] + 7   # outside the pool
    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    pa.decode_append(q.to(dev), k_new.to(dev), v_new.to(dev), kd, vd, bt_bad.to(dev),
                     sl_bad.to(dev), max_len, partition_tokens=4 * bs)
    torch.cuda.synchronize()
    err = pa.last_device_error()
    assert err & pa.DEVERR_SEQ_LEN and err & pa.DEVERR_TABLE_ENTRY
    # the oracle writes only sequences 0 and 3
    keep = torch.tensor([0, 3])
    slots = torch.from_numpy(oracle.slots_from_positions(keep.int(), sl[keep] - 1, bt, bs))
    kh, vh = kc.clone(), vc.clone()
    oracle.write_kv(k_new[keep], v_new[keep], slots, kh, vh)
    assert torch.equal(kd.cpu().view(torch.uint8), kh.view(torch.uint8))
    assert torch.equal(vd.cpu().view(torch.uint8), vh.view(torch.uint8))


@pytest.mark.parametrize("name,kw", [
    ("mha", dict(num_seqs=8, min_len=128, max_len=700, num_blocks=1024)),
    ("gqa", dict(num_seqs=24, median_len=300, max_len=2000, num_shared=6, prefix_len=128,
                 num_blocks=4096)),
    ("long", dict(num_seqs=2, seq_len=9000)),
])
def test_append_workload_steps(cuda_device, name, kw):
    """The serving workloads' decode step (one new token per sequence at its
    last position) through the one call, against the oracle's slot-mapping
    write and decode."""
    wl = workloads.make(name, **kw)
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    for st in wl.steps:
        assert torch.equal(st.seq_ids, torch.arange(wl.num_seqs, dtype=torch.int32))
        assert torch.equal(st.positions, st.seq_lens - 1)
        out = d.append(st)
        h.write(st)
        torch.cuda.synchronize()
        assert_close(out.cpu().double().numpy(), h.decode(st), BF16_ATOL, BF16_RTOL, name)
    assert torch.equal(d.k_cache.cpu(), h.k_cache) and torch.equal(d.v_cache.cpu(), h.v_cache)
    assert pa.last_device_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["long", "mha", "gqa"])
def test_append_full_size_sampled(cuda_device, name):
    """The full-size workload in the launch configuration the step loop times
    (automatic partition): the caches after the call equal the oracle's write
    on every appended row, and sampled outputs match the oracle."""
    wl = workloads.make(name)
    st = wl.steps[0]
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    out = d.append(st).cpu()
    h.write(st)
    slots = st.slot_mapping
    nb, bs = wl.num_blocks, wl.block_size
    blk, row = slots // bs, slots % bs
    assert torch.equal(d.k_cache[blk.to(cuda_device), :, row.to(cuda_device)].cpu(),
                       h.k_cache[blk, :, row])
    assert torch.equal(d.v_cache[blk.to(cuda_device), :, row.to(cuda_device)].cpu(),
                       h.v_cache[blk, :, row])
    pairs = sample_pairs(st, wl.num_q_heads, 48, seed=2)
    ref = h.decode(st, pairs=pairs)
    got = out.double().numpy()
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref[pairs[:, 0], pairs[:, 1]],
                 BF16_ATOL, BF16_RTOL, f"{name} append full")
    assert torch.isfinite(out.float()).all()
    assert pa.last_device_error() == 0
    assert nb == wl.k_cache.shape[0]


def test_append_in_a_cuda_graph(cuda_device):
    """Decode steps of one call each, captured once and replayed as the
    lengths grow: the same caches and outputs as the oracle step by step."""
    hkv, group, d, bs = 8, 4, 128, 16
    lens0 = [200, 31, 1, 500]
    steps = 5
    n = len(lens0)
    g = torch.Generator().manual_seed(13)
    width = max(-(-(t + steps) // bs) for t in lens0)
    nb = n * width + 2
    perm = torch.randperm(nb, generator=g)[:n * width].view(n, width).int()
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    kh, vh = kc.clone(), vc.clone()
    bt = perm.to(dev)
    max_len = max(lens0) + steps
    q_buf = torch.empty(n, hkv * group, d, dtype=torch.bfloat16, device=dev)
    k_buf = torch.empty(n, hkv, d, dtype=torch.bfloat16, device=dev)
    v_buf = torch.empty_like(k_buf)
    sl_buf = torch.empty(n, dtype=torch.int32, device=dev)
    out = torch.empty_like(q_buf)
    ws = torch.empty(max(pa.decode_workspace_bytes(n, hkv * group, max_len, kd), 256),
                     dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    sl_buf.copy_(torch.tensor(lens0, dtype=torch.int32))
    q_buf.zero_()
    k_buf.zero_()
    v_buf.zero_()
    with torch.cuda.stream(side):
        # warm the call on the capture stream (descriptors, attributes);
        # these rows are overwritten by the first replay
        pa.decode_append(q_buf, k_buf, v_buf, kd, vd, bt, sl_buf, max_len, out=out,
                         workspace=ws, stream=side)
        side.synchronize()
        kd.copy_(kc.to(dev))
        vd.copy_(vc.to(dev))
        with torch.cuda.graph(graph, stream=side):
            pa.decode_append(q_buf, k_buf, v_buf, kd, vd, bt, sl_buf, max_len, out=out,
                             workspace=ws, stream=side)
    torch.cuda.synchronize()
    for s in range(steps):
        lens = torch.tensor([t + s + 1 for t in lens0], dtype=torch.int32)
        q = torch.randn(n, hkv * group, d, generator=g).to(torch.bfloat16)
        kn = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16)
        vn = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16)
        q_buf.copy_(q)
        k_buf.copy_(kn)
        v_buf.copy_(vn)
        sl_buf.copy_(lens)
        graph.replay()
        torch.cuda.synchronize()
        slots = torch.from_numpy(oracle.slots_from_positions(
            torch.arange(n, dtype=torch.int32), lens - 1, perm, bs))
        oracle.write_kv(kn, vn, slots, kh, vh)
        ref = oracle.decode(q, kh, vh, perm, lens, 1 / math.sqrt(d))
        assert_close(out.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"graph step {s}")
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    assert pa.last_device_error() == 0


def test_fork_then_append_steps(cuda_device):
    """The decode loop with shared blocks: three sequences forked from a
    parent whose tail block is partly filled (ref_cnt 4), and a fifth on its
    own, take six steps.  Each step is BlockPool.append_step (copy-on-write
    of the shared tail for all but its last sharer, fresh blocks when a tail
    fills), pa_copy_blocks of its pairs, then pa_decode_append; the oracle
    replays the same copies and writes at the pool's own slots."""
    hkv, group, d, bs = 8, 4, 128, 16
    nb = 128
    pool = BlockPool(nb, bs, np.random.default_rng(1).permutation(nb))
    pool.add("P", 37)
    for c in ("c0", "c1", "c2"):
        pool.fork("P", c)
    pool.add("Q", 100)
    seqs = ["P", "c0", "c1", "c2", "Q"]
    g = torch.Generator().manual_seed(44)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    kh, vh = kc.clone(), vc.clone()
    scale = 1 / math.sqrt(d)
    copies = 0
    for step in range(6):
        pairs = pool.append_step(seqs)
        copies += len(pairs)
        if pairs:
            pt = torch.tensor(pairs, dtype=torch.int64)
            pa.copy_blocks(kd, vd, kd, vd, pt.to(dev))
            assert oracle.copy_blocks(kh, vh, kh, vh, pt) == 0
        lens = torch.tensor([pool.lengths[s] for s in seqs], dtype=torch.int32)
        bt = torch.tensor(pool.table_rows(seqs, pool.blocks_for(int(lens.max()))),
                          dtype=torch.int32)
        q = torch.randn(len(seqs), hkv * group, d, generator=g).to(torch.bfloat16)
        kn = torch.randn(len(seqs), hkv, d, generator=g).to(torch.bfloat16)
        vn = torch.randn(len(seqs), hkv, d, generator=g).to(torch.bfloat16)
        out = pa.decode_append(q.to(dev), kn.to(dev), vn.to(dev), kd, vd, bt.to(dev),
                               lens.to(dev), int(lens.max()), scale, partition_tokens=32)
        torch.cuda.synchronize()
        slots = torch.tensor([pool.slot(s, pool.lengths[s] - 1) for s in seqs],
                             dtype=torch.int64)
        assert oracle.write_kv(kn, vn, slots, kh, vh) == 0
        ref = oracle.decode(q, kh, vh, bt, lens, scale)
        assert_close(out.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"step {step}")
    assert copies == 3                                 # c0, c1, c2 copy P's tail once each
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    assert pa.last_device_error() == 0
