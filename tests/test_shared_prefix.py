"""pa_decode_shared_prefix against the oracle: groups of sequences whose
tables start with the same physical blocks (a shared prompt prefix with
ref_cnt > 1), decoded with the shared blocks read once per kv head and row
tile, must give the oracle's plain decode over the same tables: the bf16
bound 3e-3 + 1e-2 |ref|, fp32 1e-5.

Cases cover several groups, group sizes that fill several row tiles, a
shared prefix that is not a whole number of partitions, a member shorter
than the shared blocks (it sees only its own keys), a member that ends
exactly at them, a member of length 0, a group with no shared blocks, group
sizes G = 1 .. 32 query heads per kv head, head dims 64 and 128, block sizes
8, 16 and 32, and the shapes the TMA kernel does not take (plain decode)."""
import ctypes
import math

import pytest
import torch

import oracle
import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import BlockPool, workloads
from tests._gpu import BF16_ATOL, BF16_RTOL, assert_close, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clear_device_error(cuda_device):
    pa.last_device_error()
    yield


def shared_batch(hq, hkv, d, bs, groups, singles, dtype=torch.bfloat16, seed=0):
    """A batch of the groups' members and the singles in a seeded order.
    groups: [(shared blocks, [member lengths])]; a member's table is the
    group's shared blocks followed by its own.  Returns q, caches, tables,
    lengths and [(member ids, shared blocks)]."""
    g = torch.Generator().manual_seed(seed)
    seqs = []                                   # (group index or -1, length)
    for k, (_, lens) in enumerate(groups):
        seqs += [(k, t) for t in lens]
    seqs += [(-1, t) for t in singles]
    order = torch.randperm(len(seqs), generator=g).tolist()
    seqs = [seqs[j] for j in order]
    need = sum(b for b, _ in groups) + sum(
        max(0, -(-t // bs) - (groups[k][0] if k >= 0 else 0)) for k, t in seqs)
    nb = need + 5
    perm = iter(torch.randperm(nb, generator=g).tolist())
    shared = [[next(perm) for _ in range(b)] for b, _ in groups]
    rows = []
    for k, t in seqs:
        row = list(shared[k]) if k >= 0 else []
        row += [next(perm) for _ in range(max(0, -(-t // bs) - len(row)))]
        rows.append(row)
    width = max(1, max(len(r) for r in rows))
    bt = torch.tensor([r + [-1] * (width - len(r)) for r in rows], dtype=torch.int32)
    sl = torch.tensor([t for _, t in seqs], dtype=torch.int32)
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(dtype)
    q = torch.randn(len(seqs), hq, d, generator=g).to(dtype)
    members = [([i for i, (k, _) in enumerate(seqs) if k == kk], b)
               for kk, (b, _) in enumerate(groups)]
    return q, kc, vc, bt, sl, members


def run_shared(dev, q, kc, vc, bt, sl, members, scale, mode=pa.SHARED_ONCE, **kw):
    grp = pa.prefix_groups(members, q.shape[0], dev)
    kw["mode"] = mode
    out = pa.decode_shared_prefix(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                                  max(1, int(sl.max())), grp, scale, **kw)
    torch.cuda.synchronize()
    return out.cpu()


CASES = [
    # hq, hkv, d, bs, groups [(shared blocks, member lengths)], singles, partition
    (32, 8, 128, 16, [(32, [600, 513, 1500, 900, 530, 777, 2000, 513])], [100, 3000, 1], 0),
    (32, 8, 128, 16, [(8, [300, 129, 500]), (4, [70, 64, 65, 200, 33])], [50], 64),
    (8, 8, 128, 16, [(5, [81, 100, 300, 81] + [90] * 12)], [40], 32),
    (64, 8, 128, 32, [(4, [129, 200, 4000])], [8000], 0),
    (128, 8, 64, 16, [(6, [97, 200, 96, 50])], [300], 48),
    (256, 8, 128, 16, [(3, [49, 60])], [10], 16),
    (32, 8, 128, 8, [(7, [57, 100, 3])], [9], 0),
    (16, 2, 64, 16, [(2, [0, 100, 40]), (0, [20, 30])], [17], 16),
    # 101 sequences x 32 heads (3232 merge CTAs), members and plain
    # sequences side by side, 8- and 2-warp merges
    (32, 8, 128, 16, [(8, [200 + 37 * j for j in range(40)]), (4, [70 + 11 * j for j in range(30)])],
     list(range(1, 400, 13)), 64),
    (32, 8, 128, 16, [(8, [200 + 37 * j for j in range(40)]), (4, [70 + 11 * j for j in range(30)])],
     list(range(1, 400, 13)), 256),
]


@pytest.mark.parametrize("hq,hkv,d,bs,groups,singles,part", CASES)
def test_shared_prefix_decode_matches_oracle(cuda_device, hq, hkv, d, bs, groups, singles,
                                             part):
    q, kc, vc, bt, sl, members = shared_batch(hq, hkv, d, bs, groups, singles, seed=hq + bs)
    assert pa.decode_path(hq, kc) == 1
    scale = 1 / math.sqrt(d)
    out = run_shared(cuda_device, q, kc, vc, bt, sl, members, scale, partition_tokens=part)
    ref = oracle.decode(q, kc, vc, bt, sl, scale)
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "shared-prefix decode")
    assert pa.last_device_error() == 0
    again = run_shared(cuda_device, q, kc, vc, bt, sl, members, scale, partition_tokens=part)
    assert torch.equal(again, out)                 # bitwise reproducible


def test_gqa_workload_groups(cuda_device):
    """The GQA workload at reduced size: its block pool's shared-prefix groups
    (ref_cnt > 1 on the prefix blocks), decoded after the step's write."""
    wl = workloads.gqa(num_seqs=24, num_shared=8, prefix_len=256, num_blocks=4096)
    assert wl.prefix_groups and len(wl.prefix_groups[0][0]) == 8
    assert wl.prefix_groups[0][1] == 256 // wl.block_size
    st = wl.steps[0]
    dev = cuda_device
    kd, vd = wl.k_cache.to(dev), wl.v_cache.to(dev)
    pa.write_kv(st.k_new.to(dev), st.v_new.to(dev), st.slot_mapping.to(dev), kd, vd)
    kh, vh = wl.k_cache.clone(), wl.v_cache.clone()
    oracle.write_kv(st.k_new, st.v_new, st.slot_mapping, kh, vh)
    grp = pa.prefix_groups(wl.prefix_groups, wl.num_seqs, dev)
    ref = oracle.decode(st.q, kh, vh, st.block_tables, st.seq_lens, wl.scale)
    for mode in (pa.SHARED_ONCE, pa.SHARED_AUTO, pa.SHARED_PLAIN):
        out = pa.decode_shared_prefix(st.q.to(dev), kd, vd, st.block_tables.to(dev),
                                      st.seq_lens.to(dev), int(st.seq_lens.max()), grp,
                                      wl.scale, mode=mode).cpu()
        assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, f"gqa workload {mode}")
    assert pa.last_device_error() == 0


def test_groups_from_the_block_pool(cuda_device):
    """Groups found by BlockPool.shared_prefix_groups after forks and a
    prefix that is not block-aligned: the forked children share every
    block of the parent up to its last full one."""
    bs = 16
    pool = BlockPool(256, bs, torch.randperm(256, generator=torch.Generator().manual_seed(7)))
    pool.add("p", 250)                              # 15 full blocks + 10 tokens
    for c in range(3):
        pool.add(c, 250 + 40 * c, prefix_of="p", prefix_tokens=240)
    pool.release("p")
    pool.add(3, 90)
    seqs = [2, 3, 0, 1]
    groups = pool.shared_prefix_groups(seqs)
    assert groups == [([0, 2, 3], 15)]
    g = torch.Generator().manual_seed(8)
    hq, hkv, d = 32, 8, 128
    kc = torch.randn(256, hkv, bs, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(256, hkv, bs, d, generator=g).to(torch.bfloat16)
    q = torch.randn(4, hq, d, generator=g).to(torch.bfloat16)
    bt = torch.tensor(pool.table_rows(seqs), dtype=torch.int32)
    sl = torch.tensor([pool.lengths[s] for s in seqs], dtype=torch.int32)
    out = run_shared(cuda_device, q, kc, vc, bt, sl, groups, 1 / math.sqrt(d),
                     partition_tokens=64)
    ref = oracle.decode(q, kc, vc, bt, sl, 1 / math.sqrt(d))
    assert_close(out.double().numpy(), ref, BF16_ATOL, BF16_RTOL, "block pool groups")


@pytest.mark.parametrize("dtype,d,hq,hkv,bs", [(torch.float32, 128, 32, 8, 16),
                                                (torch.bfloat16, 96, 64, 8, 16),
                                                (torch.bfloat16, 96, 8, 2, 16),
                                                (torch.bfloat16, 96, 64, 8, 4)])
def test_other_shapes_run_the_plain_decode(cuda_device, dtype, d, hq, hkv, bs):
    """Shapes whose decode kernel has no shared-prefix instance (fp32, the
    CUDA-core and mma.sync kernels, the TMA kernel at head dims other than 64
    and 128) run the plain decode in every mode."""
    q, kc, vc, bt, sl, members = shared_batch(hq, hkv, d, bs, [(4, [100, 70, 65])], [30],
                                              dtype=dtype, seed=3)
    assert pa.decode_shared_prefix_mode(hq, 4, kc, pa.SHARED_ONCE) == 0
    scale = 1 / math.sqrt(d)
    out = run_shared(cuda_device, q, kc, vc, bt, sl, members, scale, partition_tokens=32)
    atol, rtol = tolerance(dtype)
    assert_close(out.double().numpy(), oracle.decode(q, kc, vc, bt, sl, scale), atol, rtol,
                 "plain decode")


def test_bad_group_id_is_reported_and_the_sequence_decoded_alone(cuda_device):
    """A seq_group entry past the groups is reported (PA_DEVERR_GROUP) and the
    sequence is decoded as one in no group; every output stays exact."""
    q, kc, vc, bt, sl, members = shared_batch(32, 8, 128, 16, [(4, [100, 90, 80])], [50],
                                              seed=4)
    dev = cuda_device
    grp = pa.prefix_groups(members, q.shape[0], dev)
    single = int((grp.seq_group == -1).nonzero()[0])
    grp.seq_group[single] = 7
    scale = 1 / math.sqrt(128)
    out = pa.decode_shared_prefix(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                                  int(sl.max()), grp, scale, partition_tokens=32,
                                  mode=pa.SHARED_ONCE).cpu()
    assert pa.last_device_error() & pa.DEVERR_GROUP
    assert_close(out.double().numpy(), oracle.decode(q, kc, vc, bt, sl, scale), BF16_ATOL,
                 BF16_RTOL, "bad group id")


def test_small_workspace_is_refused(cuda_device):
    q, kc, vc, bt, sl, members = shared_batch(32, 8, 128, 16, [(4, [100, 90])], [50], seed=5)
    dev = cuda_device
    grp = pa.prefix_groups(members, q.shape[0], dev)
    need = pa.decode_shared_prefix_workspace_bytes(q.shape[0], 32, int(sl.max()), 4, kc, 32)
    assert need >= pa.decode_workspace_bytes(q.shape[0], 32, int(sl.max()), kc, 32) > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(pa.PaError) as e:
        pa.decode_shared_prefix(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                                int(sl.max()), grp, 0.1, workspace=ws, partition_tokens=32,
                                mode=pa.SHARED_ONCE)
    assert e.value.status == pa.PA_ERR_WORKSPACE


def test_debug_pass_refuses_a_member_with_other_leading_blocks(cuda_device, monkeypatch):
    q, kc, vc, bt, sl, members = shared_batch(32, 8, 128, 16, [(4, [100, 90, 80])], [50],
                                              seed=6)
    bad = bt.clone()
    m = members[0][0][1]
    bad[m, 2] = bt[members[0][0][0], 3]            # a private block where a shared one belongs
    bad[m, 3] = bt[members[0][0][0], 2]
    monkeypatch.setenv("PA_DEBUG", "1")
    with pytest.raises(pa.PaError) as e:
        run_shared(cuda_device, q, kc, vc, bad, sl, members, 0.1)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    monkeypatch.setenv("PA_DEBUG", "0")
    out = run_shared(cuda_device, q, kc, vc, bt, sl, members, 0.1)   # the valid call still runs
    assert_close(out.double().numpy(), oracle.decode(q, kc, vc, bt, sl, 0.1), BF16_ATOL,
                 BF16_RTOL, "valid call")


def test_c_abi_group_of_one_and_no_groups(cuda_device):
    """Through the C ABI: a group of one member (allowed there) and a call
    with no groups both equal pa_decode's output."""
    lib = pa.load_library()
    q, kc, vc, bt, sl, _ = shared_batch(32, 8, 128, 16, [], [300, 70], seed=9)
    dev = cuda_device
    qd, kd, vd, btd, sld = q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev)
    ref = pa.decode(qd, kd, vd, btd, sld, 300, 0.1, partition_tokens=64)
    for members, blocks in (([1], 4), ([], 0)):
        grp = pa.prefix_groups([], 2, dev)
        if members:
            grp = pa.PrefixGroups(torch.tensor([-1, 0], dtype=torch.int32, device=dev),
                                  torch.tensor([0, 1], dtype=torch.int32, device=dev),
                                  torch.tensor(members, dtype=torch.int32, device=dev),
                                  torch.tensor([blocks], dtype=torch.int32, device=dev), 1,
                                  blocks)
        need = pa.decode_shared_prefix_workspace_bytes(2, 32, 300, grp.max_prefix_blocks, kc, 64)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        out = torch.full_like(qd, float("nan"))
        st = lib.pa_decode_shared_prefix(
            qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), btd.data_ptr(), bt.shape[1],
            sld.data_ptr(), 2, 300, 32, ctypes.c_float(0.1), 64, grp.seq_group.data_ptr(),
            grp.member_start.data_ptr(), grp.members.data_ptr() if members else None,
            grp.prefix_blocks.data_ptr() if members else None, grp.num_groups,
            grp.max_group_size, grp.max_prefix_blocks, pa.SHARED_ONCE, out.data_ptr(),
            ws.data_ptr(),
            ws.numel(), ctypes.byref(pa.cache_desc(kd)), torch.cuda.current_stream().cuda_stream)
        assert st == pa.PA_OK
        torch.cuda.synchronize()
        assert_close(out.cpu().double().numpy(), ref.cpu().double().numpy(), 2 * BF16_ATOL,
                     2 * BF16_RTOL, f"group {members}")


def test_automatic_mode_reads_once_only_where_it_pays(cuda_device):
    """The automatic choice: once when a row tile holds at least two members
    and the prefix saves at least 1024 tokens of reads per member."""
    kc = torch.empty(1, 8, 16, 128, dtype=torch.bfloat16)
    mode = lambda hq, blocks, m=pa.SHARED_AUTO: pa.decode_shared_prefix_mode(hq, blocks, kc, m)
    assert mode(32, 32) == 0            # G = 4, 512 tokens: 2 members a tile, 256 saved
    assert mode(32, 128) == 1           # 2048 tokens: 1024 saved
    assert mode(8, 128) == 1            # G = 1: 8 members a tile
    assert mode(8, 64) == 0             # 1024 tokens * 7/8 < 1024
    assert mode(64, 1024) == 0          # G = 8: one member a tile
    assert mode(32, 32, pa.SHARED_ONCE) == 1 and mode(32, 1024, pa.SHARED_PLAIN) == 0
    f32 = torch.empty(1, 8, 16, 128, dtype=torch.float32)
    assert pa.decode_shared_prefix_mode(32, 1024, f32, pa.SHARED_ONCE) == 0   # plain kernel
    assert mode(32, 32, 7) < 0


def test_debug_pass_refuses_seq_group_that_disagrees_with_members(cuda_device, monkeypatch):
    """A member not marked in seq_group, and a sequence marked but not listed,
    are refused under PA_DEBUG before launch (without it the output would be
    undefined)."""
    q, kc, vc, bt, sl, members = shared_batch(32, 8, 128, 16, [(4, [100, 90, 80])], [50],
                                              seed=13)
    dev = cuda_device
    monkeypatch.setenv("PA_DEBUG", "1")
    for bad in ("unmarked member", "marked outsider"):
        grp = pa.prefix_groups(members, q.shape[0], dev)
        if bad == "unmarked member":
            grp.seq_group[members[0][0][1]] = -1
        else:
            grp.seq_group[int((grp.seq_group == -1).nonzero()[0])] = 0
        with pytest.raises(pa.PaError) as e:
            pa.decode_shared_prefix(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                                    int(sl.max()), grp, 0.1, mode=pa.SHARED_ONCE)
        assert e.value.status == pa.PA_ERR_INVALID_ARG, bad
    assert pa.last_device_error() == 0                 # nothing was launched


def test_inconsistent_member_offsets_are_reported(cuda_device):
    """member_start entries that leave [0, member_start[num_groups]] or run
    backwards: the prefix CTAs read no member and report PA_DEVERR_GROUP;
    the sequences in no group are still exact."""
    q, kc, vc, bt, sl, members = shared_batch(32, 8, 128, 16, [(4, [100, 90]), (2, [70])], [50],
                                              seed=14)
    dev = cuda_device
    grp = pa.prefix_groups(members, q.shape[0], dev)          # one group: the [70] one is dropped
    bad = pa.PrefixGroups(grp.seq_group, torch.tensor([0, 3], dtype=torch.int32, device=dev),
                          grp.members, grp.prefix_blocks, grp.max_group_size,
                          grp.max_prefix_blocks)
    # the group claims 3 members, more than max_group_size (2): refused before
    # any member is read (members holds only 2)
    out = pa.decode_shared_prefix(q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), sl.to(dev),
                                  int(sl.max()), bad, 0.1, partition_tokens=32,
                                  mode=pa.SHARED_ONCE).cpu()
    assert pa.last_device_error() & pa.DEVERR_GROUP
    ref = oracle.decode(q, kc, vc, bt, sl, 0.1)
    alone = (grp.seq_group == -1).cpu().numpy()
    assert_close(out.double().numpy()[alone], ref[alone], BF16_ATOL, BF16_RTOL, "no-group rows")
