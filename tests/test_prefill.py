"""pa_prefill (causal multi-query paged attention) on the GPU against the
oracle: bf16 within 3e-3 + 1e-2 |ref|, fp32 within 1e-5."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import workloads
from tests._gpu import BF16_ATOL, BF16_RTOL, assert_close, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clear_device_error(cuda_device):
    pa.last_device_error()
    yield


def case(hq, hkv, d, bs, ctx, qlens, dtype=torch.bfloat16, seed=0, extra_blocks=3):
    """Sequences of total length ctx[i] whose last qlens[i] positions are queried."""
    g = torch.Generator().manual_seed(seed)
    need = [-(-t // bs) for t in ctx]
    nb = sum(need) + extra_blocks
    perm = torch.randperm(nb, generator=g).tolist()
    width = max(need)
    tables, pos = [], 0
    for k in need:
        tables.append(perm[pos:pos + k] + [-1] * (width - k))
        pos += k
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    qs = [0]
    for L in qlens:
        qs.append(qs[-1] + L)
    q = torch.randn(qs[-1], hq, d, generator=g).to(dtype)
    return (q, torch.tensor(qs, dtype=torch.int32), kc, vc,
            torch.tensor(tables, dtype=torch.int32), torch.tensor(ctx, dtype=torch.int32))


def run(dev, q, qs, kc, vc, bt, sl, scale):
    out = pa.prefill(q.to(dev), qs.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                     int((qs[1:] - qs[:-1]).max()), int(sl.max()), scale)
    torch.cuda.synchronize()
    return out.cpu()


FAST = [
    # Hq, Hkv, D, B, contexts, query lengths
    (32, 8, 128, 16, (300, 17, 64, 1000), (300, 5, 64, 100)),     # G=4: prompt, chunks
    (32, 32, 128, 16, (70, 129), (70, 33)),                       # G=1 (MHA)
    (64, 8, 128, 32, (257, 40), (100, 40)),                       # G=8, B=32
    (16, 1, 128, 16, (90,), (17,)),                               # G=16
    (8, 4, 64, 64, (130, 64, 1), (130, 7, 1)),                    # G=2, D=64, B=64
    (32, 8, 128, 8, (45, 200), (45, 31)),                         # B=8
    (32, 8, 128, 16, (5, 3, 9), (1, 1, 1)),                       # decode rows only
    (32, 8, 128, 256, (600, 300, 40), (333, 0, 40)),              # B=256; a sequence with no rows
    (32, 8, 128, 48, (200, 97), (150, 60)),                       # B=48: three boxes per block
    (16, 1, 64, 16, (77, 300), (77, 129)),                        # G=16, D=64
    (64, 2, 128, 16, (300, 41), (150, 41)),                       # G=32: 4 tokens a tile
    (64, 1, 64, 32, (90,), (90,)),                                # G=64: 2 tokens a tile
    (128, 1, 128, 16, (33, 70), (33, 20)),                        # G=128: 1 token a tile
    (28, 4, 128, 16, (300, 77), (200, 77)),                       # G=7: 18 tokens, 2 rows idle
    (40, 8, 128, 16, (150,), (150,)),                             # G=5: 25 tokens, 3 rows idle
    (24, 2, 64, 16, (61, 130), (61, 40)),                         # G=12: 10 tokens, 8 rows idle
    (32, 8, 96, 16, (300, 17, 1000), (300, 5, 100)),              # D=96 in a 128-column tile
    (32, 32, 80, 16, (70, 129), (70, 33)),                        # D=80, MHA
    (64, 8, 112, 32, (257, 40), (100, 40)),                       # D=112, G=8, B=32
    (40, 8, 96, 8, (150, 3), (150, 3)),                           # D=96, G=5, B=8
    (32, 8, 48, 16, (300, 17, 1000), (300, 5, 100)),              # D=48 in a 64-column tile
    (16, 4, 32, 32, (257, 40), (100, 40)),                        # D=32, B=32
    (8, 8, 16, 8, (45, 200), (45, 31)),                           # D=16, MHA, B=8
]


@pytest.mark.parametrize("hq,hkv,d,bs,ctx,qlens", FAST)
def test_fast_prefill_matches_oracle(cuda_device, hq, hkv, d, bs, ctx, qlens):
    q, qs, kc, vc, bt, sl = case(hq, hkv, d, bs, ctx, qlens, seed=hq + bs)
    assert pa.decode_path(hq, kc) == 1
    scale = 1 / math.sqrt(d)
    out = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    ref = oracle.prefill(q, qs, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "prefill")
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("hq,hkv,d,bs,ctx,qlens,dtype", [
    (4, 2, 8, 4, (10, 7), (10, 3), torch.float32),               # the worked-example shape
    (12, 4, 256, 16, (100, 33), (20, 33), torch.bfloat16),       # D=256: 32-row tiles
    (6, 2, 96, 8, (50,), (9,), torch.bfloat16),                  # D=96
    (32, 8, 128, 16, (300, 40), (64, 40), torch.float32),
    (32, 8, 128, 16, (2000, 700), (600, 700), torch.float32),    # many key chunks and tiles
    (12, 4, 200, 3, (300, 70), (120, 70), torch.bfloat16),       # G=3: 21 tokens a tile, 1 row idle
    (24, 2, 40, 5, (333, 7), (100, 7), torch.bfloat16),          # G=12, D=40, B=5
    (160, 2, 64, 16, (90, 20), (90, 5), torch.float32),          # G=80: two CTAs per kv head
    (8, 8, 136, 7, (129, 64), (129, 1), torch.float32),          # fp32 rows over 512 bytes
    (6, 3, 12, 16, (30, 70), (30, 9), torch.bfloat16),           # 24-byte rows: generic kernel
    (16, 8, 256, 16, (700, 300), (500, 300), torch.bfloat16),    # Gemma-like D=256, G=2: mma.sync
    (12, 4, 160, 5, (333, 64), (200, 1), torch.bfloat16),        # D=160, B=5, a decode row
    (32, 32, 80, 16, (257, 99), (257, 33), torch.bfloat16),      # D=80 MHA: 64 tokens a tile
    (160, 2, 96, 16, (90, 20), (90, 5), torch.bfloat16),         # mma.sync, G=80: two CTAs per kv head
])
def test_portable_prefill_matches_oracle(cuda_device, hq, hkv, d, bs, ctx, qlens, dtype):
    """The kernels for the shapes the tcgen05 kernel does not take: mma.sync
    (bf16, head dims that are multiples of 16), CUDA-core tiled (fp32 and the
    other bf16 head dims), generic (rows that are not whole 16-byte pieces)."""
    q, qs, kc, vc, bt, sl = case(hq, hkv, d, bs, ctx, qlens, dtype=dtype, seed=d)
    scale = 0.8 / math.sqrt(d)
    out = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    ref = oracle.prefill(q, qs, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    assert_close(out.double().numpy(), ref, atol, rtol, "portable prefill")


def test_long_context_slides_the_table_window(cuda_device):
    """A 20000-token context needs 1250 table entries: more than the kernel's
    1024-entry window."""
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (20000,), (70,), seed=3)
    scale = 1 / math.sqrt(128)
    out = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    ref = oracle.prefill(q, qs, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "long context")


def test_decode_rows_agree_with_pa_decode(cuda_device):
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (700, 30, 2000), (1, 1, 1), seed=4)
    scale = 1 / math.sqrt(128)
    out = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    dec = pa.decode(q.to(cuda_device), kc.to(cuda_device), vc.to(cuda_device),
                    bt.to(cuda_device), sl.to(cuda_device), int(sl.max()), scale).cpu()
    assert_close(out.double().numpy(), dec.double().numpy(), 2 * BF16_ATOL, 2 * BF16_RTOL,
                 "prefill vs decode")


def test_chunks_agree_with_the_whole_prompt(cuda_device):
    """Rows 60..99 of a 100-token prompt equal a 40-token chunk over the same
    cache (the chunked-prefill invariant)."""
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (100,), (100,), seed=5)
    scale = 1 / math.sqrt(128)
    whole = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    part = run(cuda_device, q[60:], torch.tensor([0, 40], dtype=torch.int32), kc, vc, bt, sl,
               scale)
    assert torch.equal(whole[60:], part) or \
        np.abs(whole[60:].double().numpy() - part.double().numpy()).max() < 2 * BF16_ATOL


def test_garbage_past_the_last_key_is_ignored(cuda_device):
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (37, 90), (5, 90), seed=6)
    scale = 1 / math.sqrt(128)
    ref = oracle.prefill(q, qs, kc, vc, bt, sl, scale)
    for i, t in enumerate(sl.tolist()):
        last = int(bt[i, (t - 1) // 16])
        kc[last, :, t % 16:] = float("nan")
        vc[last, :, t % 16:] = float("inf")
    out = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "nan tail")


def test_query_longer_than_sequence_is_reported(cuda_device):
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (40, 60), (10, 20), seed=7)
    sl = sl.clone()
    sl[0] = 5                                      # 10 query rows but only 5 positions
    out = pa.prefill(q.to(cuda_device), qs.to(cuda_device), kc.to(cuda_device),
                     vc.to(cuda_device), bt.to(cuda_device), sl.to(cuda_device), 20, 60, 0.1)
    torch.cuda.synchronize()
    assert pa.last_device_error() & pa.DEVERR_SEQ_LEN
    rest = (q[10:], torch.tensor([0, 20], dtype=torch.int32), kc, vc, bt[1:], sl[1:], 0.1)
    assert_close(out[10:].double().cpu().numpy(), oracle.prefill(*rest), BF16_ATOL, BF16_RTOL,
                 "other sequence")


def test_prefill_workload_reduced(cuda_device):
    """The chunked-prefill workload at reduced size: write the chunk, attend."""
    wl = workloads.prefill(num_seqs=3, max_len0=500, chunk=200, num_blocks=1024)
    st = wl.steps[0]
    kd, vd = wl.k_cache.to(cuda_device), wl.v_cache.to(cuda_device)
    pa.write_kv(st.k_new.to(cuda_device), st.v_new.to(cuda_device),
                st.slot_mapping.to(cuda_device), kd, vd)
    out = pa.prefill(st.q.to(cuda_device), st.query_start.to(cuda_device), kd, vd,
                     st.block_tables.to(cuda_device), st.seq_lens.to(cuda_device), 200,
                     int(st.seq_lens.max()), wl.scale).cpu()
    kh, vh = wl.k_cache.clone(), wl.v_cache.clone()
    oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kh, vh)
    args = (st.q, st.query_start, kh, vh, st.block_tables, st.seq_lens, wl.scale)
    assert_close(out.double().numpy(), oracle.prefill(*args), BF16_ATOL, BF16_RTOL,
                 "prefill workload")


def test_negative_scale_takes_the_portable_kernel(cuda_device):
    """The tcgen05 kernel needs scale >= 0; a negative scale is computed by
    the mma.sync kernel."""
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (150, 60), (40, 60), seed=8)
    out = run(cuda_device, q, qs, kc, vc, bt, sl, -0.05)
    args = (q, qs, kc, vc, bt, sl, -0.05)
    assert_close(out.double().numpy(), oracle.prefill(*args), BF16_ATOL, BF16_RTOL,
                 "negative scale")


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (4, 2, 8)])
def test_bad_table_entry_is_reported(cuda_device, hq, hkv, d):
    """An out-of-range block id in one sequence's table raises the error bit;
    the other sequence's rows are unaffected (fast and portable kernels)."""
    q, qs, kc, vc, bt, sl = case(hq, hkv, d, 16, (300, 200), (100, 50), seed=9)
    rest = (q[100:], torch.tensor([0, 50], dtype=torch.int32), kc, vc, bt[1:], sl[1:],
            1 / math.sqrt(d))
    ref = oracle.prefill(*rest)
    bad = bt.clone()
    bad[0, 3] = kc.shape[0] + 5
    out = run(cuda_device, q, qs, kc, vc, bad, sl, 1 / math.sqrt(d))
    assert pa.last_device_error() & pa.DEVERR_TABLE_ENTRY
    assert_close(out[100:].double().numpy(), ref, BF16_ATOL, BF16_RTOL, "other sequence")


def test_prefill_from_pinned_host_arguments(cuda_device):
    """q, query starts, tables, lengths and out in page-locked host memory give
    the same bits as device tensors."""
    q, qs, kc, vc, bt, sl = case(32, 8, 128, 16, (300, 90), (120, 90), seed=10)
    scale = 1 / math.sqrt(128)
    ref = run(cuda_device, q, qs, kc, vc, bt, sl, scale)
    kd, vd = kc.to(cuda_device), vc.to(cuda_device)
    out_h = torch.empty_like(q).pin_memory()
    pa.prefill(q.pin_memory(), qs.pin_memory(), kd, vd, bt.pin_memory(), sl.pin_memory(), 120,
               300, scale, out=out_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref)


@pytest.mark.slow
def test_prefill_workload_full_size_sampled(cuda_device):
    """The chunked-prefill workload at full size (8 x 2048-token chunks over
    histories up to 4096 tokens), in the configuration the bench times:
    48 sampled (row, head) outputs against the oracle.  Each sampled row r of
    sequence i at position p is the single-query attention of q[r] over the
    keys 0..p, computed by the oracle as a sequence of length p + 1."""
    wl = workloads.prefill()
    st = wl.steps[0]
    kd, vd = wl.k_cache.to(cuda_device), wl.v_cache.to(cuda_device)
    pa.write_kv(st.k_new.to(cuda_device), st.v_new.to(cuda_device),
                st.slot_mapping.to(cuda_device), kd, vd)
    qs = st.query_start
    max_q = int((qs[1:] - qs[:-1]).max())
    out = pa.prefill(st.q.to(cuda_device), qs.to(cuda_device), kd, vd,
                     st.block_tables.to(cuda_device), st.seq_lens.to(cuda_device), max_q,
                     int(st.seq_lens.max()), wl.scale).cpu()
    assert pa.last_device_error() == 0
    assert torch.isfinite(out.float()).all()
    del kd, vd
    oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, wl.k_cache, wl.v_cache)
    rng = np.random.default_rng(13)
    rows = rng.integers(0, int(qs[-1]), size=48)
    heads = rng.integers(0, wl.num_q_heads, size=48)
    seq = np.searchsorted(qs.numpy(), rows, side="right") - 1
    T, L = st.seq_lens.numpy()[seq], (qs[1:] - qs[:-1]).numpy()[seq]
    pos = T - L + (rows - qs.numpy()[seq])
    q1 = st.q[torch.from_numpy(rows)]
    bt1 = st.block_tables[torch.from_numpy(seq)]
    sl1 = torch.from_numpy((pos + 1).astype(np.int32))
    pairs = np.stack([np.arange(48), heads], axis=1)
    ref = oracle.decode(q1, wl.k_cache, wl.v_cache, bt1, sl1, wl.scale, pairs=pairs)
    got = out[torch.from_numpy(rows), torch.from_numpy(heads)].double().numpy()
    assert_close(got, ref[np.arange(48), heads], BF16_ATOL, BF16_RTOL, "prefill full size")


@pytest.mark.parametrize("d,dtype,hq,hkv", [(64, torch.float32, 8, 2), (96, torch.bfloat16, 8, 2),
                                           (128, torch.bfloat16, 32, 8)])
@pytest.mark.parametrize("shift", ["q", "out"])
def test_unaligned_query_or_output(cuda_device, d, dtype, hq, hkv, shift):
    """q or out one element off their allocation's alignment: each kernel
    takes only the alignments it can use (16-byte copies and stores), and the
    others fall back; the result is the oracle's either way."""
    q, qs, kc, vc, bt, sl = case(hq, hkv, d, 16, (200, 90), (70, 90), dtype=dtype, seed=31)
    scale = 1 / math.sqrt(d)
    dev = cuda_device

    def shifted(t):
        buf = torch.zeros(t.numel() + 1, dtype=t.dtype, device=dev)
        view = buf[1:].view(t.shape)
        view.copy_(t.to(dev))
        return view

    qd = shifted(q) if shift == "q" else q.to(dev)
    out = shifted(torch.zeros_like(q)) if shift == "out" else None
    got = pa.prefill(qd, qs.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                     int((qs[1:] - qs[:-1]).max()), int(sl.max()), scale, out=out)
    torch.cuda.synchronize()
    args = (q, qs, kc, vc, bt, sl, scale)
    atol, rtol = tolerance(dtype)
    assert_close(got.cpu().double().numpy(), oracle.prefill(*args), atol, rtol,
                 f"shifted {shift}")
    assert pa.last_device_error() == 0
