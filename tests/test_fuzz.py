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
from tests._gpu import BF16_ATOL, BF16_RTOL, F32_ATOL, assert_close, prefill_weight_rounding

pytestmark = pytest.mark.gpu

BLOCK_SIZES = (8, 16, 32, 48, 64, 128)


def _case(rng, prefill=False):
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    d = int(rng.choice([64, 128]))
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
def test_fuzz_prefill(cuda_device, seed):
    rng = np.random.default_rng(2000 + seed)
    hkv, g, d, bs, lens = _case(rng, prefill=True)
    hq = hkv * g
    kc, vc, bt, gen = _pool(rng, hkv, d, bs, lens, torch.bfloat16)
    # each sequence queries its last L_i positions (0 <= L_i <= T_i)
    qlens = [int(rng.integers(0, t + 1)) if rng.random() < 0.8 else t for t in lens]
    qs = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    total = int(qs[-1])
    if total == 0:
        qlens[0], total = 1, 1
        qs = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    q = torch.randn(total, hq, d, generator=gen).to(torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32)
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    dev = cuda_device
    out = pa.prefill(q.to(dev), qs.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                     max(qlens), max(lens), scale)
    torch.cuda.synchronize()
    ref = oracle.prefill(q, qs, kc, vc, bt, sl, scale)
    what = f"hq={hq} hkv={hkv} d={d} B={bs} lens={lens} rows={qlens}"
    # the tensor-core kernel (128 rows a tile: G divides 128) multiplies bf16 P
    extra = prefill_weight_rounding(q, qs, kc, vc, bt, sl, scale) if 128 % g == 0 else None
    assert_close(out.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, what, extra)
    assert pa.last_device_error() == 0
