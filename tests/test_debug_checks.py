"""PA_DEBUG=1: the host validation pass refuses, before any launch, what the
kernels cannot see from one CTA (two tokens on one slot, two copies into
one block) and what they would only skip and report (entries outside the
pool, lengths past their bounds).  Valid calls give the same results with the
pass on."""
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from tests._gpu import BF16_ATOL, BF16_RTOL, assert_close
from tests.test_decode import gpu_decode, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture
def debug_on(monkeypatch, cuda_device):
    pa.last_device_error()
    monkeypatch.setenv("PA_DEBUG", "1")
    yield cuda_device
    assert pa.last_device_error() == 0            # nothing was launched to report


def _refused(fn):
    with pytest.raises(pa.PaError) as e:
        fn()
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def _pool(dev, nb=16, hkv=2, bs=4, d=64, seed=0):
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16)
    return kc, vc, kc.to(dev), vc.to(dev)


def _tokens(n, hkv=2, d=64, seed=1):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, hkv, d, generator=g).to(torch.bfloat16),
            torch.randn(n, hkv, d, generator=g).to(torch.bfloat16))


def test_write_duplicate_slot_is_refused(debug_on):
    dev = debug_on
    _, _, kd, vd = _pool(dev)
    k, v = _tokens(3)
    before = kd.clone()
    slots = torch.tensor([5, 9, 5], dtype=torch.int64, device=dev)
    _refused(lambda: pa.write_kv(k.to(dev), v.to(dev), slots, kd, vd))
    assert torch.equal(kd, before)                 # nothing was written


def test_write_slot_past_pool_is_refused(debug_on):
    dev = debug_on
    _, _, kd, vd = _pool(dev)
    k, v = _tokens(2)
    slots = torch.tensor([3, 16 * 4], dtype=torch.int64, device=dev)
    _refused(lambda: pa.write_kv(k.to(dev), v.to(dev), slots, kd, vd))


def test_valid_write_is_unchanged_by_the_checks(debug_on):
    dev = debug_on
    kc, vc, kd, vd = _pool(dev)
    k, v = _tokens(4)
    slots = torch.tensor([7, -1, 0, 63], dtype=torch.int64)
    pa.write_kv(k.to(dev), v.to(dev), slots.to(dev), kd, vd)
    assert oracle.write_kv(k, v, slots, kc, vc) == 0
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)


def test_positions_that_meet_on_one_slot_are_refused(debug_on):
    dev = debug_on
    _, _, kd, vd = _pool(dev)
    k, v = _tokens(2)
    tables = torch.tensor([[3, 4], [5, 3]], dtype=torch.int32, device=dev)
    # sequence 0 position 1 and sequence 1 position 5 both land in block 3, row 1
    seq_ids = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    positions = torch.tensor([1, 5], dtype=torch.int32, device=dev)
    _refused(lambda: pa.write_kv_positions(k.to(dev), v.to(dev), seq_ids, positions, tables,
                                           kd, vd))


def test_decode_bad_needed_entry_and_long_length_are_refused(debug_on):
    dev = debug_on
    q, kc, vc, bt, sl = synthetic(8, 2, 64, 16, [40, 17])
    bad = bt.clone()
    bad[1, 1] = kc.shape[0]                        # needed by length 17: outside the pool
    _refused(lambda: gpu_decode(dev, q, kc, vc, bad, sl, 0.125))
    with pytest.raises(pa.PaError):
        pa.decode(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev), 39, 0.125)


def test_decode_unused_padding_passes_and_matches(debug_on):
    dev = debug_on
    q, kc, vc, bt, sl = synthetic(8, 2, 64, 16, [40, 17, 3])
    out = gpu_decode(dev, q, kc, vc, bt, sl, 0.125)
    ref = oracle.decode(q, kc, vc, bt, sl, 0.125)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "decode with PA_DEBUG")


def test_prefill_more_rows_than_positions_is_refused(debug_on):
    dev = debug_on
    _, kc, vc, bt, sl = synthetic(8, 2, 64, 16, [20, 9])
    qs = torch.tensor([0, 5, 15], dtype=torch.int32)      # sequence 1: 10 rows, 9 positions
    q = torch.randn(15, 8, 64).to(torch.bfloat16)
    _refused(lambda: pa.prefill(q.to(dev), qs.to(dev), kc.to(dev), vc.to(dev), bt.to(dev),
                                sl.to(dev), 10, 20))


def test_copy_into_one_block_twice_or_onto_a_source_is_refused(debug_on):
    dev = debug_on
    _, _, kd, vd = _pool(dev)
    twice = torch.tensor([[1, 7], [2, 7]], dtype=torch.int64, device=dev)
    _refused(lambda: pa.copy_blocks(kd, vd, kd, vd, twice))
    chain = torch.tensor([[1, 2], [2, 3]], dtype=torch.int64, device=dev)
    _refused(lambda: pa.copy_blocks(kd, vd, kd, vd, chain))
    outside = torch.tensor([[1, 16]], dtype=torch.int64, device=dev)
    _refused(lambda: pa.copy_blocks(kd, vd, kd, vd, outside))
    ok = torch.tensor([[1, 2], [3, 4]], dtype=torch.int64, device=dev)
    pa.copy_blocks(kd, vd, kd, vd, ok)
    torch.cuda.synchronize()
    assert torch.equal(kd[2], kd[1]) and torch.equal(vd[4], vd[3])


def test_without_pa_debug_the_pass_is_off(monkeypatch, cuda_device):
    """Without the variable a duplicate slot is the caller's error: the call
    launches (which of the two tokens lands is undefined)."""
    monkeypatch.delenv("PA_DEBUG", raising=False)
    dev = cuda_device
    _, _, kd, vd = _pool(dev)
    k, v = _tokens(2)
    slots = torch.tensor([5, 5], dtype=torch.int64, device=dev)
    pa.write_kv(k.to(dev), v.to(dev), slots, kd, vd)
    torch.cuda.synchronize()
    assert pa.last_device_error() == 0


def test_append_into_a_shared_block_is_refused(debug_on):
    """pa_decode_append whose appended slot lies in a block another table
    also reaches (not copied first) is refused before launch; the same batch
    with the block made private passes and matches the oracle."""
    import math
    dev = debug_on
    kc, vc, kd, vd = _pool(dev)
    # both sequences' tables start with block 7; sequence 0 (5 tokens, B = 4)
    # appends into its own block 3, sequence 1 (3 tokens) into block 7
    bt = torch.tensor([[7, 3], [7, -1]], dtype=torch.int32)
    sl = torch.tensor([5, 3], dtype=torch.int32)
    q = torch.randn(2, 4, 64, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    k, v = _tokens(2)
    before = kd.clone()
    _refused(lambda: pa.decode_append(q.to(dev), k.to(dev), v.to(dev), kd, vd, bt.to(dev),
                                      sl.to(dev), 8))
    assert torch.equal(kd, before)
    bt[1, 0] = 9                                        # sequence 1 on a private block
    out = pa.decode_append(q.to(dev), k.to(dev), v.to(dev), kd, vd, bt.to(dev), sl.to(dev), 8)
    torch.cuda.synchronize()
    slots = torch.from_numpy(oracle.slots_from_positions(torch.arange(2, dtype=torch.int32),
                                                         sl - 1, bt, 4))
    kh, vh = kc.clone(), vc.clone()
    oracle.write_kv(k, v, slots, kh, vh)
    ref = oracle.decode(q, kh, vh, bt, sl, 1 / math.sqrt(64))
    assert torch.equal(kd.cpu(), kh)
    assert_close(out.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, "debug append")


def test_two_appends_on_one_slot_are_refused(debug_on):
    """Two sequences whose tables end in the same block at the same offset
    (one slot appended twice) are refused; the shared-block rule names it
    first."""
    dev = debug_on
    _, _, kd, vd = _pool(dev)
    bt = torch.tensor([[2, 5], [4, 5]], dtype=torch.int32)
    sl = torch.tensor([6, 6], dtype=torch.int32)
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    k, v = _tokens(2)
    _refused(lambda: pa.decode_append(q.to(dev), k.to(dev), v.to(dev), kd, vd, bt.to(dev),
                                      sl.to(dev), 8))
