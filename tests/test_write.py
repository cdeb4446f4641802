"""pa_write_kv on the GPU against the oracle's sequential scatter: bit-exact."""
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import workloads
from tests._gpu import DeviceState, HostState

pytestmark = pytest.mark.gpu


def _random_write(dev, nb, hkv, bs, d, dtype, n_tok, seed, extra_slots=()):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(n_tok, hkv, d, generator=g).to(dtype)
    v = torch.randn(n_tok, hkv, d, generator=g).to(dtype)
    slots = torch.randperm(nb * bs, generator=g)[:n_tok].to(torch.int64)
    for pos, s in extra_slots:
        slots[pos] = s
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    kh, vh = kc.clone(), vc.clone()
    rejected = oracle.write_kv(k, v, slots, kh, vh)
    kd, vd = kc.to(dev), vc.to(dev)
    pa.write_kv(k.to(dev), v.to(dev), slots.to(dev), kd, vd)
    return kd.cpu(), vd.cpu(), kh, vh, rejected


@pytest.mark.parametrize("hkv,bs,d,dtype", [
    (8, 16, 128, torch.bfloat16), (32, 16, 128, torch.bfloat16), (8, 32, 128, torch.bfloat16),
    (2, 4, 8, torch.float32), (3, 5, 6, torch.bfloat16), (2, 3, 3, torch.float32),
    (1, 7, 1, torch.bfloat16), (4, 16, 64, torch.float32)])
def test_write_bit_exact(cuda_device, hkv, bs, d, dtype):
    kd, vd, kh, vh, rej = _random_write(cuda_device, 40, hkv, bs, d, dtype, 57, 1,
                                        extra_slots=[(3, -1), (10, -7)])
    assert rej == 0
    assert torch.equal(kd.view(torch.uint8), kh.view(torch.uint8))
    assert torch.equal(vd.view(torch.uint8), vh.view(torch.uint8))
    assert pa.last_device_error() == 0


def test_write_out_of_range_slot_is_skipped_and_reported(cuda_device):
    nb, bs = 20, 16
    kd, vd, kh, vh, rej = _random_write(cuda_device, nb, 8, bs, 128, torch.bfloat16, 30, 2,
                                        extra_slots=[(5, nb * bs), (6, nb * bs + 1000)])
    assert rej == 2
    assert torch.equal(kd, kh) and torch.equal(vd, vh)
    assert pa.last_device_error() & pa.DEVERR_SLOT
    assert pa.last_device_error() == 0          # cleared by the previous read


def test_write_empty_is_noop(cuda_device):
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device=cuda_device)
    e = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=cuda_device)
    pa.write_kv(e, e, torch.empty(0, dtype=torch.int64, device=cuda_device), kc, kc.clone())
    torch.cuda.synchronize()
    assert not kc.any()


def test_write_worked_example(cuda_device):
    wl = workloads.tiny()
    st = wl.steps[0]
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    d.write(st)
    h.write(st)
    assert torch.equal(d.k_cache.cpu(), h.k_cache) and torch.equal(d.v_cache.cpu(), h.v_cache)


def test_write_continuous_batching_steps_small(cuda_device):
    wl = workloads.cb(num_seqs=16, max_len0=300, chunk=100, num_steps=4, num_blocks=2048)
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    for st in wl.steps:
        d.write(st)
        h.write(st)
    assert torch.equal(d.k_cache.cpu(), h.k_cache) and torch.equal(d.v_cache.cpu(), h.v_cache)


@pytest.mark.slow
def test_write_continuous_batching_full_step(cuda_device):
    """Full-size step: 256 decode tokens + one 2048-token chunk (2304 rows)."""
    wl = workloads.cb(num_steps=1)
    st = wl.steps[0]
    assert st.slot_mapping.numel() == 2304
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    d.write(st)
    h.write(st)
    # compare every written block in full, and the whole cache by checksum
    blocks = torch.unique(st.slot_mapping // wl.block_size)
    assert torch.equal(d.k_cache[blocks.to(cuda_device)].cpu(), h.k_cache[blocks])
    assert torch.equal(d.v_cache[blocks.to(cuda_device)].cpu(), h.v_cache[blocks])
    hk = h.k_cache.to(cuda_device)
    assert torch.equal(d.k_cache, hk)
    del hk
    assert torch.equal(d.v_cache, h.v_cache.to(cuda_device))


@pytest.mark.parametrize("positions", [False, True])
def test_write_from_pinned_host_arguments(cuda_device, positions):
    """New K/V, slots (or ids, positions and tables) in page-locked host memory,
    read by the kernel over the host link: the caches match the oracle bit for bit."""
    nb, hkv, bs, d = 64, 8, 16, 128
    g = torch.Generator().manual_seed(31)
    n_tok = 40
    tables = torch.randperm(nb, generator=g)[:60].view(6, 10).int()
    seq_ids = torch.randint(0, 6, (n_tok,), generator=g, dtype=torch.int32)
    pos = torch.randperm(10 * bs, generator=g)[:n_tok].to(torch.int32)
    slots = torch.from_numpy(oracle.slots_from_positions(seq_ids, pos, tables, bs))
    k = torch.randn(n_tok, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(n_tok, hkv, d, generator=g).to(torch.bfloat16)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    kh, vh = kc.clone(), vc.clone()
    oracle.write_kv(k, v, slots, kh, vh)
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    if positions:
        pa.write_kv_positions(k.pin_memory(), v.pin_memory(), seq_ids.pin_memory(),
                              pos.pin_memory(), tables.pin_memory(), kd, vd)
    else:
        pa.write_kv(k.pin_memory(), v.pin_memory(), slots.pin_memory(), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    assert pa.last_device_error() == 0
