"""The library inside CUDA graphs, the way a serving loop runs its decode
steps: the write and the decode are captured once on static buffers, and
each replay after new inputs are copied in must match the oracle step by
step.  The grid is fixed at capture from the host bound max_seq_len, so
lengths may grow up to it between replays."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from tests._gpu import BF16_ATOL, BF16_RTOL, assert_close

pytestmark = pytest.mark.gpu

N, HQ, HKV, D, B = 8, 32, 8, 128, 16
POOL, WIDTH = 512, 40                       # blocks in the pool, table width (640 tokens)
MAX_LEN = WIDTH * B


def _setup(seed=0):
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(POOL, HKV, B, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(POOL, HKV, B, D, generator=g).to(torch.bfloat16)
    perm = torch.randperm(POOL, generator=g)[:N * WIDTH]
    tables = perm.view(N, WIDTH).to(torch.int32)
    base = torch.randint(1, MAX_LEN - 8, (N,), generator=g, dtype=torch.int32)
    return g, kc, vc, tables, base


def _step_inputs(g, tables, lens):
    """One decode step: a new token at position lens[i] - 1 of each sequence."""
    pos = (lens - 1).long()
    slots = tables.long().gather(1, (pos // B).unsqueeze(1)).squeeze(1) * B + pos % B
    q = torch.randn(N, HQ, D, generator=g).to(torch.bfloat16)
    k = torch.randn(N, HKV, D, generator=g).to(torch.bfloat16)
    v = torch.randn(N, HKV, D, generator=g).to(torch.bfloat16)
    return q, k, v, slots


@pytest.mark.parametrize("partition", [0, 64])
def test_write_and_decode_replay_as_one_graph(cuda_device, partition):
    dev = cuda_device
    g, kc, vc, tables, base = _setup()
    kd, vd = kc.to(dev), vc.to(dev)
    scale = 1 / math.sqrt(D)
    # static device buffers the graph reads
    q_s = torch.zeros(N, HQ, D, dtype=torch.bfloat16, device=dev)
    k_s = torch.zeros(N, HKV, D, dtype=torch.bfloat16, device=dev)
    v_s = torch.zeros_like(k_s)
    slots_s = torch.full((N,), -1, dtype=torch.int64, device=dev)   # warm-up writes nothing
    tables_s = tables.to(dev)
    lens_s = base.to(dev)

    def step():
        pa.write_kv(k_s, v_s, slots_s, kd, vd)
        return pa.decode(q_s, kd, vd, tables_s, lens_s, MAX_LEN, scale,
                         partition_tokens=partition)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()                                     # warm-up outside the capture
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out_s = step()
    torch.cuda.synchronize()
    assert pa.last_device_error() == 0

    host_k, host_v = kc.clone(), vc.clone()
    lens = base.clone()
    for s in range(4):
        lens = lens + 1                            # each sequence gains its new token
        q, k, v, slots = _step_inputs(g, tables, lens)
        for dst, src in ((q_s, q), (k_s, k), (v_s, v), (slots_s, slots), (lens_s, lens)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert oracle.write_kv(k, v, slots, host_k, host_v) == 0
        ref = oracle.decode(q, host_k, host_v, tables, lens, scale)
        assert_close(out_s.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"replay {s}")
    assert torch.equal(kd.cpu(), host_k) and torch.equal(vd.cpu(), host_v)
    assert pa.last_device_error() == 0


def test_copy_on_write_in_a_graph(cuda_device):
    """A block copy captured in a graph copies whatever the pairs buffer holds
    at replay."""
    dev = cuda_device
    _, kc, vc, _, _ = _setup(seed=1)
    kd, vd = kc.to(dev), vc.to(dev)
    pairs_s = torch.tensor([[0, 1]], dtype=torch.int64, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        pa.copy_blocks(kd, vd, kd, vd, pairs_s)
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.copy_blocks(kd, vd, kd, vd, pairs_s)
    for src, dst in ((5, 9), (100, 3), (7, 500)):
        pairs_s.copy_(torch.tensor([[src, dst]], dtype=torch.int64))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(kd[dst], kd[src]) and torch.equal(vd[dst], vd[src])
    assert pa.last_device_error() == 0


def test_back_to_back_steps_without_synchronising(cuda_device):
    """Continuous-batching steps issued back to back (each kernel may start
    before the previous one ends, by programmatic dependent launch), with no
    synchronisation until the end: every step's output and the final caches
    match the oracle replaying the same steps in order."""
    from paged_kv_cache_109_gb300 import workloads
    dev = cuda_device
    wl = workloads.make("cb", num_seqs=12, num_steps=4, num_blocks=4096)
    kd, vd = wl.k_cache.to(dev), wl.v_cache.to(dev)
    # every step's inputs on the device first: a copy from pageable memory
    # inside the loop would wait for the stream
    ds = [{k: getattr(st, k).to(dev) for k in ("q", "k_new", "v_new", "slot_mapping",
                                               "block_tables", "seq_lens")} for st in wl.steps]
    torch.cuda.synchronize()
    outs = []
    for _ in range(2):
        for st, d in zip(wl.steps, ds):
            pa.write_kv(d["k_new"], d["v_new"], d["slot_mapping"], kd, vd)
            for part in (0, 64):
                outs.append(pa.decode(d["q"], kd, vd, d["block_tables"], d["seq_lens"],
                                      int(st.seq_lens.max()), wl.scale, partition_tokens=part))
    torch.cuda.synchronize()
    assert pa.last_device_error() == 0
    kh, vh = wl.k_cache.clone(), wl.v_cache.clone()
    i = 0
    for _ in range(2):
        for st in wl.steps:
            assert oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kh, vh) == 0
            ref = oracle.decode(st.q, kh, vh, st.block_tables, st.seq_lens, wl.scale)
            for part in (0, 64):
                assert_close(outs[i].cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL,
                             f"step {i // 2} partition {part}")
                i += 1
    assert torch.equal(kd.cpu(), kh) and torch.equal(vd.cpu(), vh)


def test_shared_prefix_decode_replays_in_a_graph(cuda_device):
    """pa_decode_shared_prefix (shared blocks read once) captured on static
    buffers: each replay decodes whatever q and lengths hold at that time,
    with the groups' arrays fixed."""
    from tests.test_shared_prefix import shared_batch
    dev = cuda_device
    q, kc, vc, bt, sl, members = shared_batch(32, 8, 128, 16, [(6, [200, 150, 300, 97])],
                                              [60, 400], seed=11)
    kd, vd = kc.to(dev), vc.to(dev)
    max_len = bt.shape[1] * 16                     # the tables' reach: a host bound
    grp = pa.prefix_groups(members, q.shape[0], dev)
    need = pa.decode_shared_prefix_workspace_bytes(q.shape[0], 32, max_len, 6, kd, 64)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    q_s, lens_s, bt_s = q.to(dev), sl.to(dev), bt.to(dev)
    scale = 1 / math.sqrt(128)

    def call():
        return pa.decode_shared_prefix(q_s, kd, vd, bt_s, lens_s, max_len, grp, scale,
                                       workspace=ws, partition_tokens=64, mode=pa.SHARED_ONCE)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()                                     # warm-up outside the capture
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out_s = call()
    g = torch.Generator().manual_seed(12)
    for s in range(3):
        q2 = torch.randn(q.shape, generator=g).to(torch.bfloat16)
        lens = torch.clamp(sl - s, min=0)          # the tables cover every length up to sl
        q_s.copy_(q2)
        lens_s.copy_(lens)
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.decode(q2, kc, vc, bt, lens, scale)
        assert_close(out_s.cpu().double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"replay {s}")
    assert pa.last_device_error() == 0
