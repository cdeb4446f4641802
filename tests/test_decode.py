"""pa_decode on the GPU against the fp64 CPU oracle.

Tolerances: fp32 caches, max abs error 1e-5; bf16 caches (the oracle reads the
same bf16 values, widened exactly), |gpu - ref| <= 3e-3 + 1e-2 |ref| per
element.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import workloads
from tests._gpu import (BF16_ATOL, BF16_RTOL, F32_ATOL, DeviceState, HostState, assert_close,
                        sample_pairs, tolerance, decode_kernel)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clear_device_error(cuda_device):
    pa.last_device_error()
    yield


def run_step(wl, dev, step_index=0, **kw):
    d, h = DeviceState(wl, dev), HostState(wl)
    st = wl.steps[step_index]
    d.write(st)
    h.write(st)
    out = d.decode(st, **kw)
    torch.cuda.synchronize()
    return out.cpu(), h.decode(st), d, h


def synthetic(hq, hkv, d, bs, lengths, dtype=torch.bfloat16, seed=0, num_blocks=None,
              shuffle=True):
    """Random caches/tables for given lengths (tables from a shuffled pool)."""
    g = torch.Generator().manual_seed(seed)
    need = [-(-t // bs) for t in lengths]
    nb = num_blocks or sum(need) + 3
    perm = torch.randperm(nb, generator=g).tolist() if shuffle else list(range(nb))
    width = max(max(need), 1)
    tables, pos = [], 0
    for k in need:
        tables.append(perm[pos:pos + k] + [-1] * (width - k))
        pos += k
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    q = torch.randn(len(lengths), hq, d, generator=g).to(dtype)
    return q, kc, vc, torch.tensor(tables, dtype=torch.int32), torch.tensor(lengths,
                                                                            dtype=torch.int32)


def gpu_decode(dev, q, kc, vc, bt, sl, scale, **kw):
    out = pa.decode(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                    int(sl.max()) if sl.numel() else 0, scale, **kw)
    torch.cuda.synchronize()
    return out.cpu()


# ---- the worked example (fp32, portable kernel) ------------------------------

def test_worked_example_fp32(cuda_device):
    wl = workloads.tiny()
    assert pa.decode_path(4, wl.k_cache) == 0
    out, ref, d, h = run_step(wl, cuda_device)
    assert_close(out.double().numpy(), ref, F32_ATOL, 0.0, "tiny")
    # paged == contiguous: dense attention on the contiguous K/V
    for s in range(2):
        ek = wl.contiguous_k[s].double().repeat_interleave(2, dim=0)
        ev = wl.contiguous_v[s].double().repeat_interleave(2, dim=0)
        for hh in range(4):
            dense = torch.softmax(ek[hh] @ wl.steps[0].q[s, hh].double() * wl.scale, 0) @ ev[hh]
            assert np.abs(out[s, hh].double().numpy() - dense.numpy()).max() <= F32_ATOL
    assert pa.last_device_error() == 0


# ---- TMA + tensor-core kernel, small ragged cases ------------------------------

FAST_CASES = [
    # (Hq, Hkv, D, B, lengths)
    (32, 32, 128, 16, (1, 15, 16, 17, 63, 64, 65, 200)),         # MHA, G=1
    (32, 8, 128, 16, (1, 5, 129, 300, 1000, 47)),                  # G=4
    (64, 8, 128, 32, (1, 31, 32, 33, 700, 1500)),                  # G=8, B=32
    (16, 1, 128, 16, (3, 77, 512)),                                # G=16
    (12, 3, 128, 16, (40, 9, 333)),                                # G=4, odd head count
    (10, 2, 64, 32, (1, 64, 65, 250)),                             # G=5, D=64
    (8, 4, 64, 64, (1, 63, 64, 65, 129, 400)),                     # G=2, B=64
    (9, 1, 64, 16, (2, 100)),                                      # G=9
    (32, 8, 128, 48, (1, 47, 48, 49, 300)),                        # B=48: 3 chunks/block
    (32, 8, 128, 128, (5, 127, 128, 129, 1000)),                   # B=128
    (64, 8, 128, 64, (64, 65, 777)),                               # G=8, B=64
    (32, 8, 128, 8, (1, 7, 8, 9, 15, 16, 17, 300)),                # B=8: 2 blocks/chunk
    (16, 16, 64, 8, (3, 24, 25, 130)),                             # B=8, D=64, MHA
    (32, 8, 128, 256, (1, 255, 256, 257, 2000)),                   # B=256: 16 chunks/block
    (32, 2, 64, 32, (1, 95, 96, 97, 800)),                         # G=16, D=64, B=32
    (64, 2, 128, 16, (5, 300, 1000)),                              # G=32: two sub-groups of 16
    (48, 2, 128, 16, (1, 17, 700)),                                # G=24: sub-groups of 16 and 8
    (40, 1, 64, 32, (33, 400)),                                    # G=40: 16, 16 and 8
    (40, 8, 96, 16, (1, 100, 257, 1500)),                          # D=96: box 2 half zero-filled
    (64, 8, 80, 32, (1, 31, 32, 33, 900)),                         # D=80, G=8, B=32
    (32, 8, 112, 16, (17, 400, 2049)),                             # D=112, G=4
    (128, 8, 96, 16, (5, 700)),                                    # D=96, G=16
    (8, 8, 96, 8, (1, 9, 130)),                                    # D=96 MHA, B=8
    (64, 8, 48, 32, (1, 31, 32, 33, 900)),                         # D=48: one box, 16 columns zero
    (32, 2, 48, 16, (1, 17, 700)),                                 # D=48, G=16
    (16, 4, 16, 16, (1, 15, 16, 17, 400)),                         # D=16: one k-step
    (32, 8, 32, 8, (1, 7, 8, 9, 300)),                             # D=32, B=8
    (8, 8, 32, 64, (63, 64, 65, 500)),                             # D=32 MHA, B=64
    (48, 2, 16, 16, (5, 333)),                                     # D=16, G=24: sub-groups
    (32, 8, 256, 16, (1, 15, 16, 17, 300, 2049)),                  # D=256: four boxes, G=4
    (64, 8, 256, 32, (33, 700, 4000)),                             # D=256, G=8, B=32
    (16, 8, 256, 8, (9, 300)),                                     # D=256, G=2, B=8
    (32, 1, 256, 16, (100, 1, 900)),                               # D=256, G=32: sub-groups
]


@pytest.mark.parametrize("hq,hkv,d,bs,lengths", FAST_CASES)
@pytest.mark.parametrize("part", [0, "B", "3B", "4B", "64B"])
def test_fast_kernel_matches_oracle(cuda_device, hq, hkv, d, bs, lengths, part):
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, bs, lengths, seed=hq * 7 + bs)
    assert pa.decode_path(hq, kc) == 1
    scale = 1.0 / math.sqrt(d)
    ptok = 0 if part == 0 else bs * int(part[:-1] or 1)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=ptok)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"fast {hq}/{hkv}/{d}/{bs}")
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("hq,hkv,d,bs,lengths,dtype", [
    (8, 2, 8, 4, (10, 7, 1, 33), torch.float32),
    (32, 8, 128, 16, (1, 200, 1000), torch.float32),
    (64, 2, 96, 24, (5, 300), torch.bfloat16),            # G=32, D=96, B=24: mma.sync
    (6, 2, 96, 12, (1, 8, 9, 100), torch.bfloat16),      # D=96, B=12: CUDA cores
    (4, 4, 256, 16, (17, 64), torch.bfloat16),           # D=256
])
@pytest.mark.parametrize("part", [0, "B", "5B"])
def test_portable_kernel_matches_oracle(cuda_device, hq, hkv, d, bs, lengths, dtype, part):
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, bs, lengths, dtype=dtype, seed=d + bs)
    assert pa.decode_path(hq, kc) == decode_kernel(dtype, d, bs, hq // hkv)
    scale = 0.9 / math.sqrt(d)
    ptok = 0 if part == 0 else bs * int(part[:-1] or 1)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=ptok)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    assert_close(out.double().numpy(), ref, atol, rtol, "portable")


@pytest.mark.parametrize("hq,hkv,d,bs,lengths,dtype,part", [
    (12, 4, 200, 3, (1, 50, 257), torch.bfloat16, 0),      # 8-token chunks, 8 columns a lane
    (12, 4, 200, 3, (1, 50, 257), torch.bfloat16, 21),     # partitions not whole chunks
    (24, 2, 40, 5, (7, 333), torch.bfloat16, 0),           # G=12: sub-groups of 8 and 4
    (24, 2, 40, 5, (7, 333), torch.bfloat16, 35),
    (8, 8, 136, 7, (100, 1, 64), torch.float32, 0),        # fp32 rows over 256 bytes
    (6, 2, 64, 1, (1100, 3), torch.float32, 1100),          # >512 blocks in one partition
    (6, 3, 12, 16, (30, 70), torch.bfloat16, 0),           # 24-byte rows: the generic kernel
    (6, 3, 12, 16, (30, 70), torch.bfloat16, 32),
    (40, 8, 96, 24, (1, 100, 257), torch.bfloat16, 0),     # mma.sync, G=5 (lo parts in rows 8-15)
    (64, 8, 48, 24, (1, 100, 257), torch.bfloat16, 48),    # mma.sync, D=48, B=24
    (96, 8, 80, 5, (700, 33), torch.bfloat16, 35),         # mma.sync, G=12, B=5
    (64, 4, 64, 1, (1100, 3), torch.bfloat16, 1100),       # mma.sync, G=16, >512 blocks a partition
    (256, 8, 112, 24, (500, 1, 90), torch.bfloat16, 0),    # mma.sync, G=32: two sub-groups
])
def test_cuda_core_kernels_match_oracle(cuda_device, hq, hkv, d, bs, lengths, dtype, part):
    """The CUDA-core kernels' own cases: chunk sizes, sub-groups, block sizes
    that split chunks into several copies, a partition whose table entries do
    not fit the kernel's shared copy, and rows that are not whole 16-byte
    pieces."""
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, bs, lengths, dtype=dtype, seed=d * 7 + bs)
    assert pa.decode_path(hq, kc) == decode_kernel(dtype, d, bs, hq // hkv)
    scale = 1.1 / math.sqrt(d)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=part)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    assert_close(out.double().numpy(), ref, atol, rtol, f"{hq}/{hkv}/{d}/{bs}/{dtype}/{part}")
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("dtype,d,bs,part,hq", [(torch.float32, 64, 16, 64, 8),
                                                (torch.bfloat16, 96, 4, 0, 8),
                                                (torch.float32, 32, 1, 1024, 8),
                                                (torch.bfloat16, 96, 4, 0, 16),
                                                (torch.bfloat16, 64, 1, 1024, 32)])
def test_bad_table_entry_on_cuda_core_kernel(cuda_device, dtype, d, bs, part, hq):
    """Out-of-range entries are reported and their tokens skipped, from the
    partition's shared copy of the table and (blocks of one token, partition
    of 1024) from the table itself; CUDA-core and mma.sync kernels."""
    q, kc, vc, bt, sl = synthetic(hq, 2, d, bs, (700, 300), dtype=dtype, seed=12)
    assert pa.decode_path(hq, kc) == decode_kernel(dtype, d, bs, hq // 2)
    bt = bt.clone()
    nb = kc.shape[0]
    bt[0, 5] = nb            # == num_blocks: out of range
    bt[1, 2] = -3
    gpu_decode(cuda_device, q, kc, vc, bt, sl, 0.1, partition_tokens=part)
    assert pa.last_device_error() & pa.DEVERR_TABLE_ENTRY


# ---- split-K partials and merge --------------------------------------------------

@pytest.mark.parametrize("hq,hkv,d,bs,part", [(32, 8, 128, 16, 64), (64, 8, 128, 32, 256),
                                               (8, 2, 8, 4, 8)])
def test_workspace_partials_match_oracle(cuda_device, hq, hkv, d, bs, part):
    dtype = torch.float32 if d == 8 else torch.bfloat16
    lengths = (1, part - 1, part, part + 1, 5 * part + 3)
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, bs, lengths, dtype=dtype, seed=5)
    scale = 1.0 / math.sqrt(d)
    n = len(lengths)
    maxlen = int(sl.max())
    need = pa.decode_workspace_bytes(n, hq, maxlen, kc, part)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=cuda_device)
    out = pa.decode(q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device),
                    bt.to(cuda_device), sl.to(cuda_device), maxlen, scale, workspace=ws,
                    partition_tokens=part)
    torch.cuda.synchronize()
    P = -(-maxlen // part)
    cells = n * hq * P
    acc = ws[: cells * d * 4].view(torch.float32).view(n, hq, P, d).cpu().double().numpy()
    off = (cells * d * 4 + 255) // 256 * 256
    ml = ws[off: off + cells * 8].view(torch.float32).view(n, hq, P, 2).cpu().double().numpy()
    m_ref, l_ref, acc_ref = oracle.decode_partials(q, kc, vc, bt, sl, scale, part, P)
    atol, rtol = tolerance(dtype)
    for s, t in enumerate(lengths):
        parts = -(-t // part)
        if parts <= 1:
            continue
        m_gpu = ml[s, :, :parts, 0] / math.log2(math.e)
        assert_close(m_gpu, m_ref[s, :, :parts], 1e-4, 1e-5, "m")
        assert_close(ml[s, :, :parts, 1], l_ref[s, :, :parts], 1e-4, 1e-3, "l")
        # acc grows with l (up to the partition length): compare acc / l,
        # the partition's own normalised output, at the output tolerance
        assert_close(acc[s, :, :parts] / ml[s, :, :parts, 1:],
                     acc_ref[s, :, :parts] / l_ref[s, :, :parts, None], atol, rtol, "acc/l")
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    assert_close(out.cpu().double().numpy(), ref, atol, rtol, "merged out")


def test_split_on_off_agree_and_runs_are_deterministic(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (3000, 1, 777, 4096, 2048), seed=9)
    scale = 1 / math.sqrt(128)
    outs = [gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=p)
            for p in (16, 64, 256, 1024, 4096)]
    for o in outs[1:]:
        assert_close(o.double().numpy(), outs[0].double().numpy(), 2 * BF16_ATOL, 2 * BF16_RTOL,
                     "split sizes")
    again = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=256)
    assert torch.equal(again, outs[2])
    auto1 = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale)
    auto2 = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale)
    assert torch.equal(auto1, auto2)


@pytest.mark.parametrize("dtype,d,hq,hkv", [(torch.bfloat16, 128, 32, 8),
                                             (torch.float32, 64, 8, 4)])
def test_many_partitions_merge(cuda_device, dtype, d, hq, hkv):
    """More partitions than the merge stages per pass (>512 here), and the
    few-partition path, on both kernels."""
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, 16, (9000, 33, 17 * 16 + 5), dtype=dtype, seed=15)
    scale = 1 / math.sqrt(d)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    for part in (16, 48, 560):
        out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=part)
        assert_close(out.double().numpy(), ref, atol, rtol, f"partitions of {part}")


@pytest.mark.parametrize("dtype,d,hq,hkv", [(torch.float32, 10, 4, 2),
                                             (torch.float32, 256, 8, 2),
                                             (torch.bfloat16, 96, 16, 2),
                                             (torch.bfloat16, 160, 8, 8)])
def test_merge_column_slabs_and_warp_counts(cuda_device, dtype, d, hq, hkv):
    """The merge on head dims that are not a multiple of 4 (one column per
    lane), wider than one 128-column slab, and at partition sizes whose
    longest sequence needs 2, 4 and 8 merge warps, with short sequences
    (fewer partitions than warps) in the same batch."""
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, 16, (2000, 40, 16 * 33, 16 * 65 + 1),
                                  dtype=dtype, seed=21)
    scale = 1 / math.sqrt(d)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    for part in (16, 32, 64):          # 125, 63 and 32 partitions in the longest sequence
        out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=part)
        assert_close(out.double().numpy(), ref, atol, rtol, f"partitions of {part}")
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("dtype,d,hq,hkv", [(torch.bfloat16, 128, 12, 4),
                                             (torch.float32, 64, 12, 4)])
def test_merge_with_thousands_of_pairs(cuda_device, dtype, d, hq, hkv):
    """A batch of 3972 (sequence, head) pairs, more merge CTAs than fit on the
    GPU at once, at partition sizes that give 2, 4 and 8 merge warps a pair,
    with pairs that need no merge next to pairs that do."""
    rng = np.random.default_rng(31)
    lens = [1, 64, 65, 1100, 0] + rng.integers(1, 1100, size=326).tolist()
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, 16, lens, dtype=dtype, seed=31)
    scale = 1 / math.sqrt(d)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    for part in (16, 64, 128, 512):    # 69, 18, 9 and 3 partitions in the longest sequence
        out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=part)
        assert_close(out.double().numpy(), ref, atol, rtol, f"partitions of {part}")
        assert torch.equal(out, gpu_decode(cuda_device, q, kc, vc, bt, sl, scale,
                                           partition_tokens=part))
    assert pa.last_device_error() == 0


def test_relabelling_physical_blocks_changes_nothing(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (500, 33, 1200), seed=3, num_blocks=200)
    scale = 1 / math.sqrt(128)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=128)
    perm = torch.randperm(200, generator=torch.Generator().manual_seed(4))
    kp, vp = torch.empty_like(kc), torch.empty_like(vc)
    kp[perm], vp[perm] = kc, vc
    btp = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    out2 = gpu_decode(cuda_device, q, kp, vp, btp, sl, scale, partition_tokens=128)
    assert torch.equal(out, out2)


def test_closed_forms_on_gpu(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (1, 100, 900), seed=6)
    scale = 1 / math.sqrt(128)
    # constant V rows -> that constant; q = 0 -> mean of V; T = 1 -> v_0
    out = gpu_decode(cuda_device, q, kc, torch.full_like(vc, 0.75), bt, sl, scale)
    assert torch.all(out == 0.75)
    out = gpu_decode(cuda_device, torch.zeros_like(q), kc, vc, bt, sl, scale)
    ref = oracle.decode(torch.zeros_like(q), kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "q=0")
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale)
    v0 = vc[int(bt[0, 0])].repeat_interleave(4, dim=0)[:, 0]        # [Hq, D]
    assert torch.equal(out[0], v0)


def test_garbage_in_unused_tail_rows_is_ignored(cuda_device):
    """Rows past T_i in a sequence's last block are never weighted, even when
    they hold NaN or Inf."""
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (37, 5, 200), seed=14)
    ref = oracle.decode(q, kc, vc, bt, sl, 1 / math.sqrt(128))
    for i, t in enumerate(sl.tolist()):
        last = int(bt[i, (t - 1) // 16])
        kc[last, :, t % 16:] = float("nan")
        vc[last, :, t % 16:] = float("inf")
    for part in (0, 16, 64):
        out = gpu_decode(cuda_device, q, kc, vc, bt, sl, 1 / math.sqrt(128),
                         partition_tokens=part)
        assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "nan tail")


def test_zero_length_sequences(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (0, 50, 0, 300), seed=8)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, 1 / math.sqrt(128), partition_tokens=64)
    assert not out[0].any() and not out[2].any()
    ref = oracle.decode(q, kc, vc, bt, sl, 1 / math.sqrt(128))
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "zero-length")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_batch_of_empty_sequences(cuda_device, dtype):
    """Every length 0 (a host bound of 0): zero rows from pa_decode and
    pa_decode_append, no cache row written, nothing reported."""
    q, kc, vc, bt, sl = synthetic(8, 2, 64, 16, (0, 0, 0), dtype=dtype, seed=9)
    dev = cuda_device
    q = q + 1                                          # nonzero queries
    out = gpu_decode(dev, q, kc, vc, bt, sl, 0.125)
    assert out.shape == q.shape and not out.any()
    kd, vd = kc.to(dev), vc.to(dev)
    k_new = torch.ones(3, 2, 64, dtype=dtype, device=dev)
    out2 = pa.decode_append(q.to(dev), k_new, k_new, kd, vd, bt.to(dev), sl.to(dev), 0, 0.125)
    torch.cuda.synchronize()
    assert not out2.any()
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    assert pa.last_device_error() == 0


# ---- device-side bounds checks (host-planted bad inputs; nothing faults) --------

def test_bad_table_entry_is_reported_not_faulting(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (100, 200), seed=10, num_blocks=40)
    bt = bt.clone()
    bt[1, 3] = 40            # == num_blocks: out of range
    bt[0, 1] = -5
    gpu_decode(cuda_device, q, kc, vc, bt, sl, 0.1, partition_tokens=64)
    assert pa.last_device_error() & pa.DEVERR_TABLE_ENTRY


def test_seq_len_beyond_bound_is_reported(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (100, 200), seed=11)
    out = pa.decode(q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device),
                    bt.to(cuda_device), sl.to(cuda_device), 150, 0.1)
    torch.cuda.synchronize()
    assert pa.last_device_error() & pa.DEVERR_SEQ_LEN
    assert torch.isfinite(out.float()).all()


def test_workspace_too_small_is_refused(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (1000, 2000), seed=12)
    ws = torch.empty(16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(pa.PaError) as e:
        pa.decode(q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device),
                  bt.to(cuda_device), sl.to(cuda_device), 2000, 0.1, workspace=ws,
                  partition_tokens=64)
    assert e.value.status == pa.PA_ERR_WORKSPACE


def test_bad_partition_is_refused(cuda_device):
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (100,), seed=13)
    with pytest.raises(pa.PaError) as e:
        pa.decode(q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device),
                  bt.to(cuda_device), sl.to(cuda_device), 100, 0.1, partition_tokens=24)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


# ---- serving-shaped workloads: reduced sizes in full, full sizes sampled ----------

@pytest.mark.parametrize("name,kw", [
    ("mha", dict(num_seqs=8, min_len=128, max_len=700, num_blocks=1024)),
    ("gqa", dict(num_seqs=24, median_len=300, max_len=2000, num_shared=6, prefix_len=128,
                 num_blocks=4096)),
    ("long", dict(num_seqs=2, seq_len=9000)),
])
def test_workload_reduced(cuda_device, name, kw):
    wl = workloads.make(name, **kw)
    out, ref, _, _ = run_step(wl, cuda_device)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, name)
    assert pa.last_device_error() == 0


def test_continuous_batching_reduced(cuda_device):
    wl = workloads.cb(num_seqs=32, max_len0=600, chunk=256, num_steps=4, num_blocks=4096)
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    for st in wl.steps:
        d.write(st)
        h.write(st)
        out = d.decode(st)
        torch.cuda.synchronize()
        assert_close(out.cpu().double().numpy(), h.decode(st), BF16_ATOL, BF16_RTOL, "cb")
    assert torch.equal(d.k_cache.cpu(), h.k_cache)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mha", "gqa", "long"])
def test_workload_full_size_sampled(cuda_device, name):
    wl = workloads.make(name)
    st = wl.steps[0]
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    d.write(st)
    h.write(st)
    out = d.decode(st).cpu()
    pairs = sample_pairs(st, wl.num_q_heads, 48, seed=1)
    ref = h.decode(st, pairs=pairs)
    got = out.double().numpy()
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref[pairs[:, 0], pairs[:, 1]],
                 BF16_ATOL, BF16_RTOL, f"{name} full")
    assert torch.isfinite(out.float()).all()
    assert pa.last_device_error() == 0
    if name == "gqa":
        assert wl.stats["prefix_ref_cnt"] == 32


@pytest.mark.slow
def test_continuous_batching_full_size_sampled(cuda_device):
    wl = workloads.cb()
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    for k, st in enumerate(wl.steps):
        d.write(st)
        h.write(st)
        out = d.decode(st).cpu()
        if k in (0, len(wl.steps) - 1):
            pairs = sample_pairs(st, wl.num_q_heads, 32, seed=k)
            ref = h.decode(st, pairs=pairs)
            got = out.double().numpy()
            assert_close(got[pairs[:, 0], pairs[:, 1]], ref[pairs[:, 0], pairs[:, 1]],
                         BF16_ATOL, BF16_RTOL, f"cb step {k}")
    assert pa.last_device_error() == 0


def test_pinned_host_step_arguments(cuda_device):
    """q, tables, lengths and out in page-locked host memory (read and written
    by the kernel over the host link) give the same bits as device tensors."""
    hq, hkv, d, bs = 32, 8, 128, 16
    g = torch.Generator().manual_seed(21)
    lens = [700, 33, 1500, 1]
    need = [-(-t // bs) for t in lens]
    nb = sum(need) + 4
    perm = torch.randperm(nb, generator=g).tolist()
    width, pos, rows = max(need), 0, []
    for k in need:
        rows.append(perm[pos:pos + k] + [-1] * (width - k))
        pos += k
    bt = torch.tensor(rows, dtype=torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16).to(cuda_device)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16).to(cuda_device)
    q = torch.randn(len(lens), hq, d, generator=g).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    ref = pa.decode(q.to(cuda_device), kc, vc, bt.to(cuda_device), sl.to(cuda_device), 1500,
                    scale, partition_tokens=256).cpu()
    out_h = torch.empty_like(q).pin_memory()
    pa.decode(q.pin_memory(), kc, vc, bt.pin_memory(), sl.pin_memory(), 1500, scale,
              out=out_h, partition_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref)
    assert pa.last_device_error() == 0


def test_pageable_or_host_cache_arguments_are_refused(cuda_device):
    import ctypes
    kc, vc, bt, sl, q = (t.to(cuda_device) for t in (
        torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16), torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16),
        torch.zeros(1, 4, dtype=torch.int32), torch.ones(1, dtype=torch.int32),
        torch.zeros(1, 4, 64, dtype=torch.bfloat16)))
    lib = pa.load_library()
    desc = pa.cache_desc(kc)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream().cuda_stream
    pageable_q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    st = lib.pa_decode(pageable_q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), 4,
                       sl.data_ptr(), 1, 16, 4, ctypes.c_float(0.1), 0, out.data_ptr(), None, 0,
                       ctypes.byref(desc), stream)
    assert st == pa.PA_ERR_INVALID_ARG
    pinned_cache = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16).pin_memory()
    st = lib.pa_decode(q.data_ptr(), pinned_cache.data_ptr(), vc.data_ptr(), bt.data_ptr(), 4,
                       sl.data_ptr(), 1, 16, 4, ctypes.c_float(0.1), 0, out.data_ptr(), None, 0,
                       ctypes.byref(desc), stream)
    assert st == pa.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("part", [256, 64])
def test_repeated_calls_on_one_workspace(cuda_device, part):
    """Split-K into 16 and 63 partitions: repeated calls on one workspace give
    the same bits, and the merged output matches the oracle."""
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (3000, 1, 777, 4000, 2048), seed=11)
    n, hq, maxlen = 5, 32, 4000
    need = pa.decode_workspace_bytes(n, hq, maxlen, kc, part)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    args = (q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device), bt.to(cuda_device),
            sl.to(cuda_device), maxlen, 1 / math.sqrt(128))
    first = pa.decode(*args, workspace=ws, partition_tokens=part).clone()
    for _ in range(3):
        again = pa.decode(*args, workspace=ws, partition_tokens=part)
        assert torch.equal(again, first)
    ref = oracle.decode(q, kc, vc, bt, sl, 1 / math.sqrt(128))
    assert_close(first.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, "merged")
    assert pa.last_device_error() == 0


def test_stale_workspace_contents_do_not_matter(cuda_device):
    """The workspace needs no initialisation: one full of 0xFF, then the same
    buffer reused by a call of another shape, both give correct outputs."""
    q, kc, vc, bt, sl = synthetic(32, 8, 128, 16, (3000, 2048, 900), seed=12)
    need = pa.decode_workspace_bytes(3, 32, 3000, kc, 256)
    ws = torch.full((need * 2,), 0xFF, dtype=torch.uint8, device=cuda_device)
    scale = 1 / math.sqrt(128)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    out = pa.decode(q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device), bt.to(cuda_device),
                    sl.to(cuda_device), 3000, scale, workspace=ws, partition_tokens=256)
    assert_close(out.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, "0xFF workspace")
    out2 = pa.decode(q[:2].to(cuda_device), kc.to(cuda_device), vc.to(cuda_device),
                     bt[:2].to(cuda_device), sl[:2].to(cuda_device), 3000, scale, workspace=ws,
                     partition_tokens=512)
    assert_close(out2.cpu().double().numpy(), ref[:2], BF16_ATOL, BF16_RTOL, "reused workspace")
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [(32, 8, 128, 16, torch.bfloat16),   # TMA
                                              (64, 8, 96, 4, torch.bfloat16),     # mma.sync
                                              (16, 8, 96, 4, torch.bfloat16),     # tiled
                                              (64, 8, 96, 16, torch.bfloat16),    # TMA, D=96
                                              (8, 2, 64, 16, torch.float32)])     # tiled fp32
@pytest.mark.parametrize("shift", ["q", "out"])
def test_unaligned_query_or_output(cuda_device, hq, hkv, d, bs, dtype, shift):
    """q or out one element off their allocation's alignment: each kernel
    takes only the alignments it can use, the others fall back, and the
    result is the oracle's either way."""
    q, kc, vc, bt, sl = synthetic(hq, hkv, d, bs, (300, 77, 1000), dtype=dtype, seed=41)
    scale = 1 / math.sqrt(d)
    dev = cuda_device

    def shifted(t):
        buf = torch.zeros(t.numel() + 1, dtype=t.dtype, device=dev)
        view = buf[1:].view(t.shape)
        view.copy_(t.to(dev))
        return view

    qd = shifted(q) if shift == "q" else q.to(dev)
    out = shifted(torch.zeros_like(q)) if shift == "out" else None
    for part in (0, 64):
        got = pa.decode(qd, kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev), int(sl.max()), scale,
                        out=out, partition_tokens=part)
        torch.cuda.synchronize()
        atol, rtol = tolerance(dtype)
        assert_close(got.cpu().double().numpy(), oracle.decode(q, kc, vc, bt, sl, scale), atol,
                     rtol, f"shifted {shift}, partition {part}")
    assert pa.last_device_error() == 0


@pytest.mark.slow
def test_million_token_sequences(cuda_device):
    """Two sequences of 2^20 tokens (1 GiB of K/V): the automatic partition
    for very long sequences (its cap rises with the length: about 300
    partitions a sequence, the merge's many-partition path) and an explicit
    partition at the largest whole-table slice, against the oracle on every
    (sequence, head)."""
    T, bs, hkv, g, d = 1 << 20, 16, 2, 4, 64
    q, kc, vc, bt, sl = synthetic(hkv * g, hkv, d, bs, (T, T - 5), seed=77)
    scale = 1 / math.sqrt(d)
    part = pa.decode_partition_tokens(2, hkv * g, T, kc)
    assert part > 1024                                  # the long-sequence cap
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    for p in (0, 2048 * bs):
        out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=p)
        assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"million tokens, {p}")
    assert pa.last_device_error() == 0


# ---- the launch's limits ------------------------------------------------------------

def test_most_sequences_one_call_takes(cuda_device):
    """65535 sequences (the grid's z limit) of 1 to 40 tokens, through
    pa_decode and pa_decode_append, against the oracle on every output; one
    more is refused before launch."""
    n = 65535
    rng = np.random.default_rng(65535)
    lens = rng.integers(1, 41, size=n).tolist()
    q, kc, vc, bt, sl = synthetic(2, 1, 64, 16, lens, seed=65)
    scale = 1 / math.sqrt(64)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "65535 sequences")
    dev = cuda_device
    g = torch.Generator().manual_seed(66)
    k_new = torch.randn(n, 1, 64, generator=g).to(torch.bfloat16)
    v_new = torch.randn(n, 1, 64, generator=g).to(torch.bfloat16)
    kd, vd = kc.to(dev), vc.to(dev)
    out2 = pa.decode_append(q.to(dev), k_new.to(dev), v_new.to(dev), kd, vd, bt.to(dev),
                            sl.to(dev), 40, scale)
    torch.cuda.synchronize()
    slots = torch.from_numpy(oracle.slots_from_positions(torch.arange(n, dtype=torch.int32),
                                                         sl - 1, bt, 16))
    kh, vh = kc.clone(), vc.clone()
    oracle.write_kv(k_new, v_new, slots, kh, vh)
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)
    ref2 = oracle.decode(q, kh, vh, bt, sl, scale)
    assert_close(out2.cpu().double().numpy(), ref2, BF16_ATOL, BF16_RTOL, "65535 appends")
    assert pa.last_device_error() == 0
    q1 = torch.zeros(n + 1, 2, 64, dtype=torch.bfloat16, device=dev)
    bt1 = torch.zeros(n + 1, bt.shape[1], dtype=torch.int32, device=dev)
    sl1 = torch.ones(n + 1, dtype=torch.int32, device=dev)
    with pytest.raises(pa.PaError) as e:
        pa.decode(q1, kd, vd, bt1, sl1, 40, scale)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_most_partitions_one_sequence_takes(cuda_device):
    """One sequence of 16 * 65535 tokens in 16-token partitions: 65535
    partials per head, the most a call takes, merged against the oracle; a
    bound of one more partition is refused before launch."""
    T = 16 * 65535
    q, kc, vc, bt, sl = synthetic(8, 1, 64, 16, (T, 3), seed=67)
    scale = 1 / math.sqrt(64)
    out = gpu_decode(cuda_device, q, kc, vc, bt, sl, scale, partition_tokens=16)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "65535 partitions")
    assert pa.last_device_error() == 0
    dev = cuda_device
    wide = torch.full((2, bt.shape[1] + 1), -1, dtype=torch.int32)
    wide[:, :bt.shape[1]] = bt
    with pytest.raises(pa.PaError) as e:
        pa.decode(q.to(dev), kc.to(dev), vc.to(dev), wide.to(dev), sl.to(dev), T + 16, scale,
                  partition_tokens=16)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
