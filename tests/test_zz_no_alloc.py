"""pa_decode_no_alloc: decode for callers that cannot allocate device memory
when they run attention (an engine's plugin hook that forbids allocation
during execution, or a process with a fixed memory budget).  It keeps the
split-K workspace in a fixed array inside libpa.so instead of taking one from
the caller.

Checked through the C ABI against pa_decode with a caller-owned workspace:
the two run the same kernels on the same arguments, so the outputs must be
equal bit for bit.  Three calls in a row (case 1, case 2, case 1 again) with
different workspace layouts: the third call must reproduce the first exactly,
whatever the second left in the shared array.  Also the size and partition
limits.  This file is collected last on purpose.
"""
import ctypes
import math

import pytest
import torch

import paged_kv_cache_109_gb300 as pa

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20      # PA_NO_ALLOC_WORKSPACE_BYTES in include/pa.h


def _fn(lib):
    f = lib.pa_decode_no_alloc
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, P, P, I32, P, I32, I32, I32, ctypes.c_float, I32, P,
                  ctypes.POINTER(pa.CacheDesc), P]
    f.restype = ctypes.c_int
    return f


def _case(dev, seed, lengths, hq=32, hkv=8, d=128, bs=16):
    g = torch.Generator().manual_seed(seed)
    need = [-(-t // bs) for t in lengths]
    nb = sum(need) + 5
    perm = torch.randperm(nb, generator=g).tolist()
    width = max(need)
    tables, pos = [], 0
    for k in need:
        tables.append(perm[pos:pos + k] + [-1] * (width - k))
        pos += k
    kc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn(nb, hkv, bs, d, generator=g).to(torch.bfloat16).to(dev)
    q = torch.randn(len(lengths), hq, d, generator=g).to(torch.bfloat16).to(dev)
    bt = torch.tensor(tables, dtype=torch.int32, device=dev)
    sl = torch.tensor(lengths, dtype=torch.int32, device=dev)
    return q, kc, vc, bt, sl


def _no_alloc(f, q, kc, vc, bt, sl, max_len, part, out):
    desc = pa.cache_desc(kc)
    return f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1],
             sl.data_ptr(), q.shape[0], max_len, q.shape[1], 1.0 / math.sqrt(q.shape[2]), part,
             out.data_ptr(), ctypes.byref(desc), torch.cuda.current_stream().cuda_stream)


def test_no_alloc_matches_pa_decode_on_calls_in_a_row(cuda_device):
    f = _fn(pa.load_library())
    cases = [(_case(cuda_device, 1, (3000, 17, 1, 900, 2049)), 256),
             (_case(cuda_device, 2, (40, 5000, 700)), 64)]
    got = []
    for (q, kc, vc, bt, sl), part in (cases[0], cases[1], cases[0]):
        max_len = int(sl.max())
        assert 0 < pa.decode_workspace_bytes(q.shape[0], q.shape[1], max_len, kc, part) <= LIMIT
        ref = pa.decode(q, kc, vc, bt, sl, max_len, partition_tokens=part)
        out = torch.full_like(q, float("nan"))
        assert _no_alloc(f, q, kc, vc, bt, sl, max_len, part, out) == pa.PA_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "no-alloc output differs from pa_decode's"
        got.append(out)
    # the replayed first case after the second left another layout in the array
    assert torch.equal(got[2], got[0])
    assert pa.last_device_error() == 0


def test_no_alloc_rejects_requests_beyond_its_array(cuda_device):
    f = _fn(pa.load_library())
    q, kc, vc, bt, sl = _case(cuda_device, 3, (64,))
    # a shape whose workspace exceeds the fixed array (4096 partitions of 16
    # tokens, within the grid's limit): refused, nothing launched
    huge_len = 1 << 16
    need = pa.decode_workspace_bytes(1024, 32, huge_len, kc, 16)
    assert need > LIMIT
    out = torch.zeros_like(q)
    st = f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(),
           1024, huge_len, 32, 0.1, 16, out.data_ptr(), ctypes.byref(pa.cache_desc(kc)),
           torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()


def test_no_alloc_refuses_more_than_65535_partitions(cuda_device):
    f = _fn(pa.load_library())
    q, kc, vc, bt, sl = _case(cuda_device, 4, (64,))
    out = torch.zeros_like(q)
    # 2^31 - 1 tokens in 16-token partitions: far more partitions than a grid takes
    st = f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), (1 << 31) // 16,
           sl.data_ptr(), 1, (1 << 31) - 1, 32, 0.1, 16, out.data_ptr(),
           ctypes.byref(pa.cache_desc(kc)), torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not out.any()
