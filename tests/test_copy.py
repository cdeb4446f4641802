"""pa_copy_blocks (copy-on-write, swapping) and pa_write_kv_positions on the
GPU against the oracle: bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300.block_pool import BlockPool
from tests._gpu import BF16_ATOL, BF16_RTOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clear_device_error(cuda_device):
    pa.last_device_error()
    yield


def _caches(nb, hkv, bs, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(nb, hkv, bs, d, generator=g).to(dtype),
            torch.randn(nb, hkv, bs, d, generator=g).to(dtype))


@pytest.mark.parametrize("hkv,bs,d,dtype", [(8, 16, 128, torch.bfloat16),
                                            (2, 4, 8, torch.float32),
                                            (3, 5, 6, torch.bfloat16)])
def test_copy_within_one_pool(cuda_device, hkv, bs, d, dtype):
    kc, vc = _caches(40, hkv, bs, d, dtype, 1)
    pairs = torch.tensor([[3, 10], [7, 11], [0, 39], [25, 12]], dtype=torch.int64)
    kh, vh = kc.clone(), vc.clone()
    assert oracle.copy_blocks(kh, vh, kh, vh, pairs) == 0
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    pa.copy_blocks(kd, vd, kd, vd, pairs.to(cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu().view(torch.uint8), kh.view(torch.uint8))
    assert torch.equal(vd.cpu().view(torch.uint8), vh.view(torch.uint8))
    assert pa.last_device_error() == 0


def test_bad_pairs_are_skipped_and_reported(cuda_device):
    kc, vc = _caches(10, 8, 16, 128, torch.bfloat16, 2)
    pairs = torch.tensor([[1, 2], [10, 3], [4, -1], [5, 6]], dtype=torch.int64)
    kh, vh = kc.clone(), vc.clone()
    assert oracle.copy_blocks(kh, vh, kh, vh, pairs) == 2
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    pa.copy_blocks(kd, vd, kd, vd, pairs.to(cuda_device))
    assert pa.last_device_error() & pa.DEVERR_BLOCK_PAIR
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)


def test_swap_out_and_in_through_pinned_host_memory(cuda_device):
    """Swap a sequence's blocks to a page-locked host pool and back."""
    nb, hkv, bs, d = 64, 8, 16, 128
    kc, vc = _caches(nb, hkv, bs, d, torch.bfloat16, 3)
    gpu_pool = BlockPool(nb, bs, np.random.default_rng(0).permutation(nb))
    host_pool = BlockPool(32, bs)
    gpu_pool.add("s", 300)                                  # 19 blocks
    table_before = list(gpu_pool.tables["s"])
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    hk = torch.zeros(32, hkv, bs, d, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = torch.tensor(gpu_pool.swap_out("s", host_pool), dtype=torch.int64)
    pa.copy_blocks(kd, vd, hk, hv, out_pairs.to(cuda_device))
    torch.cuda.synchronize()
    for gb, hb in out_pairs.tolist():
        assert torch.equal(hk[hb], kc[gb]) and torch.equal(hv[hb], vc[gb])
    # the device blocks are reused meanwhile, then the sequence comes back
    kd[table_before] = 0
    vd[table_before] = 0
    in_pairs = torch.tensor(gpu_pool.swap_in("s", host_pool), dtype=torch.int64).pin_memory()
    pa.copy_blocks(hk, hv, kd, vd, in_pairs)                # pairs read from host memory too
    torch.cuda.synchronize()
    for (hb, gb), old in zip(in_pairs.tolist(), table_before):
        assert torch.equal(kd[gb].cpu(), kc[old]) and torch.equal(vd[gb].cpu(), vc[old])
    assert pa.last_device_error() == 0


def test_pageable_host_memory_is_refused(cuda_device):
    kd, vd = (t.to(cuda_device) for t in _caches(4, 2, 16, 64, torch.bfloat16, 4))
    pageable = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device=cuda_device)
    lib = pa.load_library()
    desc = pa.cache_desc(kd)
    import ctypes
    st = lib.pa_copy_blocks(kd.data_ptr(), vd.data_ptr(), 4, pageable.data_ptr(),
                            pageable.data_ptr(), 4, pairs.data_ptr(), 1, ctypes.byref(desc),
                            torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_INVALID_ARG
    assert not pageable.any()


def test_copy_on_write_then_decode(cuda_device):
    """Branches share a partly filled tail; one branch writes after its
    copy-on-write; every branch's output matches the oracle."""
    hq, hkv, d, bs = 32, 8, 128, 16
    nb = 256
    kc, vc = _caches(nb, hkv, bs, d, torch.bfloat16, 5)
    pool = BlockPool(nb, bs, np.random.default_rng(1).permutation(nb))
    pool.add("p", 100)                                       # 7 blocks, tail holds 4 rows
    for c in range(3):
        pool.fork("p", c)
    pool.release("p")
    pairs = []
    for c in (0, 1):                                         # the last branch writes in place
        pr = pool.copy_on_write(c)
        assert pr is not None
        pairs.append(pr)
    assert pool.copy_on_write(2) is None
    g = torch.Generator().manual_seed(6)
    k_new = torch.randn(3, hkv, d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(3, hkv, d, generator=g).to(torch.bfloat16)
    slots = []
    for c in range(3):
        pool.grow(c, 1)
        slots.append(pool.slot(c, 100))
    slots = torch.tensor(slots, dtype=torch.int64)
    seqs = [0, 1, 2]
    bt = torch.tensor(pool.table_rows(seqs, 8), dtype=torch.int32)
    sl = torch.tensor([101] * 3, dtype=torch.int32)
    q = torch.randn(3, hq, d, generator=g).to(torch.bfloat16)
    # oracle
    kh, vh = kc.clone(), vc.clone()
    oracle.copy_blocks(kh, vh, kh, vh, pairs)
    oracle.write_kv(k_new, v_new, slots, kh, vh)
    ref = oracle.decode(q, kh, vh, bt, sl, 1 / math.sqrt(d))
    # device
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    pa.copy_blocks(kd, vd, kd, vd, torch.tensor(pairs, dtype=torch.int64, device=cuda_device))
    pa.write_kv(k_new.to(cuda_device), v_new.to(cuda_device), slots.to(cuda_device), kd, vd)
    out = pa.decode(q.to(cuda_device), kd, vd, bt.to(cuda_device), sl.to(cuda_device), 101)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    assert_close(out.double().cpu().numpy(), ref, BF16_ATOL, BF16_RTOL, "cow decode")


@pytest.mark.parametrize("hkv,bs,d,dtype", [(8, 16, 128, torch.bfloat16),
                                            (2, 4, 8, torch.float32)])
def test_write_by_position_matches_slot_mapping(cuda_device, hkv, bs, d, dtype):
    nb = 64
    g = torch.Generator().manual_seed(7)
    tables = torch.randperm(nb, generator=g)[:40].view(5, 8).int()
    tables[4, 5:] = -1                                      # a padded row
    seq_ids = torch.tensor([0, 0, 3, 4, 4, -1, 2, 6, 4, 1], dtype=torch.int32)
    positions = torch.tensor([0, 17, 5, 3, 80, 2, -4, 1, 8 * bs + 2, 31], dtype=torch.int32)
    # token 4: position 80 // bs may hit the padded entries of row 4 (B=16 -> entry 5)
    # token 7: sequence 6 does not exist; token 8: past the table
    n = seq_ids.numel()
    k = torch.randn(n, hkv, d, generator=g).to(dtype)
    v = torch.randn(n, hkv, d, generator=g).to(dtype)
    kc, vc = _caches(nb, hkv, bs, d, dtype, 8)
    slots = torch.from_numpy(oracle.slots_from_positions(seq_ids, positions, tables, bs))
    kh, vh = kc.clone(), vc.clone()
    oracle.write_kv(k, v, slots, kh, vh)
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    pa.write_kv_positions(k.to(cuda_device), v.to(cuda_device), seq_ids.to(cuda_device),
                          positions.to(cuda_device), tables.to(cuda_device), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu().view(torch.uint8), kh.view(torch.uint8))
    assert torch.equal(vd.cpu().view(torch.uint8), vh.view(torch.uint8))
    assert pa.last_device_error() & pa.DEVERR_TABLE_ENTRY     # tokens 7 and 8 (and 4 if padded)


def test_continuous_batching_write_by_position(cuda_device):
    """The continuous-batching steps written with device-side slots leave the
    caches bit-identical to the oracle's slot-mapping writes."""
    from paged_kv_cache_109_gb300 import workloads
    wl = workloads.cb(num_seqs=16, max_len0=300, chunk=100, num_steps=3, num_blocks=2048)
    kd, vd = wl.k_cache.to(cuda_device), wl.v_cache.to(cuda_device)
    kh, vh = wl.k_cache.clone(), wl.v_cache.clone()
    for st in wl.steps:
        oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kh, vh)
        pa.write_kv_positions(st.k_new.to(cuda_device), st.v_new.to(cuda_device),
                              st.seq_ids.to(cuda_device), st.positions.to(cuda_device),
                              st.block_tables.to(cuda_device), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    assert pa.last_device_error() == 0
