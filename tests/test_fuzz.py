"""Seeded random shapes against the oracle: decode and prefill over the
kernels' whole supported range (group size, head dim, block size, lengths
including zero, partition sizes), with the write step in front.  Each case is
small enough for the oracle; the seeds are fixed, so a failure names its case."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from tests._gpu import BF16_ATOL, BF16_RTOL, F32_ATOL, assert_close, decode_kernel

pytestmark = pytest.mark.gpu

BLOCK_SIZES = (8, 16, 32, 48, 64, 128)


def _case(rng, prefill=False):
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 24, 32]))
    d = int(rng.choice([16, 32, 48, 64, 80, 96, 112, 128, 256]))
    bs = int(rng.choice(BLOCK_SIZES))
    n = int(rng.integers(1, 7))
    lens = rng.integers(0 if not prefill else 1, 700, size=n)
    if rng.random() < 0.3:
        lens[rng.integers(n)] = int(rng.integers(1, 4))          # a very short sequence
    return hkv, g, d, bs, [int(x) for x in lens]


def _pool(rng, hkv, d, bs, lens, dtype, spare=5):
    need = [-(-t // bs) for t in lens]
    nb = sum(need) + spare
    perm = rng.permutation(nb)
    width = max(max(need), 1)
    tables, pos = [], 0
    for k in need:
        tables.append(list(perm[pos:pos + k]) + [-1] * (width - k))
        pos += k
    g = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    return kc, vc, torch.tensor(tables, dtype=torch.int32), g


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_write_then_decode(cuda_device, seed):
    rng = np.random.default_rng(1000 + seed)
    hkv, g, d, bs, lens = _case(rng)
    hq = hkv * g
    dtype = torch.float32 if rng.random() < 0.15 else torch.bfloat16
    kc, vc, bt, gen = _pool(rng, hkv, d, bs, lens, dtype)
    sl = torch.tensor(lens, dtype=torch.int32)
    # one new token per non-empty sequence, at its last position
    pos = [t - 1 for t in lens if t > 0]
    seqs = [i for i, t in enumerate(lens) if t > 0]
    slots = torch.tensor([int(bt[i, p // bs]) * bs + p % bs for i, p in zip(seqs, pos)],
                         dtype=torch.int64)
    k_new = torch.randn(len(seqs), hkv, d, generator=gen).to(dtype)
    v_new = torch.randn(len(seqs), hkv, d, generator=gen).to(dtype)
    q = torch.randn(len(lens), hq, d, generator=gen).to(dtype)
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    part = 0 if rng.random() < 0.5 else bs * int(rng.integers(1, 9))

    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    if seqs:
        pa.write_kv(k_new.to(dev), v_new.to(dev), slots.to(dev), kd, vd)
        assert oracle.write_kv(k_new, v_new, slots, kc, vc) == 0
    max_len = max(max(lens), 1)
    out = pa.decode(q.to(dev), kd, vd, bt.to(dev), sl.to(dev), max_len, scale,
                    partition_tokens=part)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = (F32_ATOL, 0.0) if dtype == torch.float32 else (BF16_ATOL, BF16_RTOL)
    what = f"hq={hq} hkv={hkv} d={d} B={bs} lens={lens} part={part} {dtype}"
    assert_close(out.cpu().double().numpy(), ref, atol, rtol, what)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_decode_append(cuda_device, seed):
    """The decode step in one call (pa_decode_append) on random shapes: its
    caches equal the oracle's write of each sequence's last position, its
    output the oracle's decode, and both equal pa_write_kv_positions +
    pa_decode bit for bit.  The appended slots hold NaN before the call."""
    rng = np.random.default_rng(3000 + seed)
    hkv, g, d, bs, lens = _case(rng)
    hq = hkv * g
    dtype = torch.float32 if rng.random() < 0.15 else torch.bfloat16
    kc, vc, bt, gen = _pool(rng, hkv, d, bs, lens, dtype)
    n = len(lens)
    for i, t in enumerate(lens):
        if t > 0:
            kc[int(bt[i, (t - 1) // bs]), :, (t - 1) % bs] = float("nan")
            vc[int(bt[i, (t - 1) // bs]), :, (t - 1) % bs] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    k_new = torch.randn(n, hkv, d, generator=gen).to(dtype)
    v_new = torch.randn(n, hkv, d, generator=gen).to(dtype)
    q = torch.randn(n, hq, d, generator=gen).to(dtype)
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    part = 0 if rng.random() < 0.5 else bs * int(rng.integers(1, 9))
    max_len = max(max(lens), 1)

    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    out = pa.decode_append(q.to(dev), k_new.to(dev), v_new.to(dev), kd, vd, bt.to(dev),
                           sl.to(dev), max_len, scale, partition_tokens=part)
    kr, vr = kc.to(dev), vc.to(dev)
    pa.write_kv_positions(k_new.to(dev), v_new.to(dev),
                          torch.arange(n, dtype=torch.int32, device=dev), (sl - 1).to(dev),
                          bt.to(dev), kr, vr)
    ref_gpu = pa.decode(q.to(dev), kr, vr, bt.to(dev), sl.to(dev), max_len, scale,
                        partition_tokens=part)
    torch.cuda.synchronize()
    slots = torch.from_numpy(oracle.slots_from_positions(
        torch.arange(n, dtype=torch.int32), sl - 1, bt, bs))
    assert oracle.write_kv(k_new, v_new, slots, kc, vc) == 0
    what = f"hq={hq} hkv={hkv} d={d} B={bs} lens={lens} part={part} {dtype}"
    assert torch.equal(kd.cpu().view(torch.uint8), kc.view(torch.uint8)), what
    assert torch.equal(vd.cpu().view(torch.uint8), vc.view(torch.uint8)), what
    assert torch.equal(kr, kd) and torch.equal(vr, vd), what
    assert torch.equal(out.view(torch.uint8), ref_gpu.view(torch.uint8)), what
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = (F32_ATOL, 0.0) if dtype == torch.float32 else (BF16_ATOL, BF16_RTOL)
    assert_close(out.cpu().double().numpy(), ref, atol, rtol, what)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_prefill(cuda_device, seed):
    rng = np.random.default_rng(2000 + seed)
    hkv, g, d, bs, lens = _case(rng, prefill=True)
    hq = hkv * g
    dtype = torch.float32 if rng.random() < 0.15 else torch.bfloat16
    kc, vc, bt, gen = _pool(rng, hkv, d, bs, lens, dtype)
    # each sequence queries its last L_i positions (0 <= L_i <= T_i)
    qlens = [int(rng.integers(0, t + 1)) if rng.random() < 0.8 else t for t in lens]
    qs = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    total = int(qs[-1])
    if total == 0:
        qlens[0], total = 1, 1
        qs = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    q = torch.randn(total, hq, d, generator=gen).to(dtype)
    sl = torch.tensor(lens, dtype=torch.int32)
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    dev = cuda_device
    out = pa.prefill(q.to(dev), qs.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                     max(qlens), max(lens), scale)
    torch.cuda.synchronize()
    ref = oracle.prefill(q, qs, kc, vc, bt, sl, scale)
    what = f"hq={hq} hkv={hkv} d={d} B={bs} lens={lens} rows={qlens} {dtype}"
    if dtype == torch.float32:                     # the portable kernel, fp32 throughout
        assert_close(out.cpu().double().numpy(), ref, F32_ATOL, 0.0, what)
    else:
        assert_close(out.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, what)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_write_from_positions(cuda_device, seed):
    """Slots computed on the device from (sequence, position): bit-exact
    against the oracle, with skipped tokens (id or position -1)."""
    rng = np.random.default_rng(3000 + seed)
    hkv, _, d, bs, lens = _case(rng, prefill=True)
    dtype = torch.float32 if rng.random() < 0.2 else torch.bfloat16
    kc, vc, bt, gen = _pool(rng, hkv, d, bs, lens, dtype)
    # distinct (sequence, position) pairs inside the lengths, a few skipped
    cand = [(i, p) for i, t in enumerate(lens) for p in range(t)]
    pick = rng.choice(len(cand), size=min(len(cand), int(rng.integers(1, 300))), replace=False)
    sid = np.array([cand[j][0] for j in pick], dtype=np.int32)
    pos = np.array([cand[j][1] for j in pick], dtype=np.int32)
    skip = rng.random(len(pick)) < 0.1
    sid[skip & (rng.random(len(pick)) < 0.5)] = -1
    pos[skip & (sid >= 0)] = -1
    k = torch.randn(len(pick), hkv, d, generator=gen).to(dtype)
    v = torch.randn(len(pick), hkv, d, generator=gen).to(dtype)
    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    pa.write_kv_positions(k.to(dev), v.to(dev), torch.from_numpy(sid).to(dev),
                          torch.from_numpy(pos).to(dev), bt.to(dev), kd, vd)
    slots = oracle.slots_from_positions(sid, pos, bt, bs)
    assert oracle.write_kv(k, v, torch.from_numpy(slots), kc, vc) == 0
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_copy_blocks(cuda_device, seed):
    """Whole-block copies inside one pool and through page-locked host memory:
    bit-exact against the oracle."""
    rng = np.random.default_rng(4000 + seed)
    hkv = int(rng.choice([1, 2, 8]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice(BLOCK_SIZES))
    nb = int(rng.integers(8, 200))
    dtype = torch.float32 if rng.random() < 0.2 else torch.bfloat16
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    n = int(rng.integers(1, nb // 2 + 1))
    perm = rng.permutation(nb)
    pairs = torch.from_numpy(np.stack([perm[:n], perm[n:2 * n]], 1).astype(np.int64))
    dev = cuda_device
    kd, vd = kc.to(dev), vc.to(dev)
    pa.copy_blocks(kd, vd, kd, vd, pairs.to(dev))
    assert oracle.copy_blocks(kc, vc, kc, vc, pairs) == 0
    # out to a pinned host pool and back into the device pool, reversed
    hk = torch.zeros(n, hkv, bs, d, dtype=dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = torch.stack([pairs[:, 1], torch.arange(n)], 1)
    back_pairs = torch.stack([torch.arange(n), pairs[:, 0]], 1)
    pa.copy_blocks(kd, vd, hk, hv, out_pairs.to(dev))
    pa.copy_blocks(hk, hv, kd, vd, back_pairs.to(dev))
    hk_ref, hv_ref = torch.zeros(n, hkv, bs, d, dtype=dtype), torch.zeros(n, hkv, bs, d, dtype=dtype)
    assert oracle.copy_blocks(kc, vc, hk_ref, hv_ref, out_pairs) == 0
    assert oracle.copy_blocks(hk_ref, hv_ref, kc, vc, back_pairs) == 0
    torch.cuda.synchronize()
    assert torch.equal(hk, hk_ref) and torch.equal(hv, hv_ref)
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_portable_shapes(cuda_device, seed):
    """Shapes the portable kernels take: head dims other than 64 and 128, fp32,
    and (prefill) groups of more than 16 query heads; decode and prefill
    against the oracle."""
    rng = np.random.default_rng(5000 + seed)
    hkv = int(rng.choice([1, 2]))
    g = int(rng.choice([1, 4, 24, 32]))
    d = int(rng.choice([8, 12, 32, 40, 96, 200, 256])) if g <= 16 else int(rng.choice([64, 96, 128]))
    bs = int(rng.choice([3, 4, 5, 8, 16, 32]))
    lens = [int(x) for x in rng.integers(1, 400, size=int(rng.integers(1, 5)))]
    hq = hkv * g
    dtype = torch.float32 if rng.random() < 0.4 else torch.bfloat16
    kc, vc, bt, gen = _pool(rng, hkv, d, bs, lens, dtype)
    assert pa.decode_path(hq, kc) == decode_kernel(dtype, d, bs, g)
    sl = torch.tensor(lens, dtype=torch.int32)
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    atol, rtol = (F32_ATOL, 0.0) if dtype == torch.float32 else (BF16_ATOL, BF16_RTOL)
    dev = cuda_device
    q = torch.randn(len(lens), hq, d, generator=gen).to(dtype)
    out = pa.decode(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev), max(lens), scale)
    torch.cuda.synchronize()
    what = f"hq={hq} hkv={hkv} d={d} B={bs} lens={lens} {dtype}"
    assert_close(out.cpu().double().numpy(), oracle.decode(q, kc, vc, bt, sl, scale), atol, rtol,
                 "decode " + what)
    qlens = [int(rng.integers(1, t + 1)) for t in lens]
    qs = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    qp = torch.randn(int(qs[-1]), hq, d, generator=gen).to(dtype)
    outp = pa.prefill(qp.to(dev), qs.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                      max(qlens), max(lens), scale)
    torch.cuda.synchronize()
    assert_close(outp.cpu().double().numpy(), oracle.prefill(qp, qs, kc, vc, bt, sl, scale),
                 atol, rtol, "prefill " + what)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_shared_prefix_decode(cuda_device, seed):
    """Random groups sharing leading blocks (sizes, shared block counts,
    members shorter than the shared blocks, sequences in no group), group
    sizes, head dims, block sizes and partitions: the shared-prefix decode
    with the shared blocks read once against the oracle's plain decode."""
    from tests.test_shared_prefix import run_shared, shared_batch
    rng = np.random.default_rng(5000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8, 16, 32]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([8, 16, 32, 64]))
    groups = []
    for _ in range(int(rng.integers(1, 4))):
        blocks = int(rng.integers(0, 11))
        lens = [int(rng.integers(0, blocks * bs + 300)) for _ in range(int(rng.integers(1, 7)))]
        groups.append((blocks, lens))
    singles = [int(rng.integers(1, 700)) for _ in range(int(rng.integers(0, 5)))]
    if max(max(lens) for _, lens in groups) == 0 and not singles:
        singles = [5]
    q, kc, vc, bt, sl, members = shared_batch(hkv * g, hkv, d, bs, groups, singles, seed=seed)
    part = 0 if rng.random() < 0.5 else bs * int(rng.integers(1, 9))
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    out = run_shared(cuda_device, q, kc, vc, bt, sl, members, scale, partition_tokens=part)
    what = f"hq={hkv * g} hkv={hkv} d={d} B={bs} groups={groups} singles={singles} part={part}"
    assert_close(out.double().numpy(), oracle.decode(q, kc, vc, bt, sl, scale), BF16_ATOL,
                 BF16_RTOL, what)
    assert pa.last_device_error() == 0
