"""The C-ABI library builds, loads and exports every symbol include/pa.h
declares; host-only entry points behave without a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "pa.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pa_write_kv", "pa_decode", "pa_decode_workspace_bytes",
                     "pa_decode_partition_tokens", "pa_decode_path", "pa_status_str",
                     "pa_last_device_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libpa.so does not export {name}"


def test_status_strings(lib):
    for code in range(5):
        s = lib.pa_status_str(code).decode()
        assert s and s != "unknown status"
    assert lib.pa_status_str(99).decode() == "unknown status"


def desc(nb=64, bs=16, hkv=8, d=128, dtype=pa.PA_BF16):
    return pa.CacheDesc(nb, bs, hkv, d, dtype)


def test_path_selection(lib):
    path = lambda hq, dd: lib.pa_decode_path(hq, ctypes.byref(dd))
    assert path(32, desc()) == 1                       # bf16, D=128, B=16, G=4
    assert path(64, desc(bs=32)) == 1                  # G=8, B=32
    assert path(128, desc(bs=32)) == 1                 # G=16
    assert path(256, desc()) == 1                      # G=32: two 16-head sub-groups
    assert path(32, desc(dtype=pa.PA_F32)) == 0        # fp32: portable kernel
    assert path(32, desc(bs=64)) == 1                  # B=64: four 16-token chunks
    assert path(32, desc(bs=48)) == 1
    assert path(32, desc(bs=8)) == 1                   # B=8: two blocks per chunk
    assert path(32, desc(bs=24)) == 0                  # neither 8 nor a multiple of 16, G=4
    assert path(32, desc(bs=4)) == 0
    assert path(32, desc(bs=512)) == 0
    assert path(64, desc(bs=24)) == 2                  # G=8: mma.sync
    assert path(64, desc(bs=4)) == 2
    assert path(40, desc(d=96)) == 1                   # D=96: two 64-column boxes
    assert path(32, desc(d=80, bs=8)) == 1
    assert path(128, desc(d=112, bs=32)) == 1
    assert path(40, desc(d=96, bs=24)) == 2            # G=5 at a block size TMA does not take
    assert path(64, desc(d=48)) == 1                   # D=48: one box, 16 columns zero-filled
    assert path(8, desc(d=16, bs=8)) == 1              # D=16, B=8
    assert path(32, desc(d=32, bs=64)) == 1
    assert path(64, desc(d=48, bs=24)) == 2            # D=48 at a block size TMA does not take
    assert path(32, desc(d=96, bs=24)) == 0            # G=4: CUDA cores
    assert path(64, desc(d=40)) == 0                   # not a multiple of 16: CUDA cores
    assert path(64, desc(d=256)) == 1                  # D=256, G=8: four boxes, one CTA a SM
    assert path(8, desc(d=256)) == 0                   # D=256, G=1: CUDA cores
    assert path(64, desc(d=192)) == 0                  # other head dims over 128: CUDA cores
    assert path(16, desc(d=64, bs=64, hkv=4)) == 1
    assert path(8, desc(d=8, bs=4, hkv=2, dtype=pa.PA_F32)) == 0
    assert path(30, desc()) == -1                      # Hq not a multiple of Hkv
    assert path(32, desc(dtype=7)) == -1


def test_workspace_layout(lib):
    d = desc(nb=16384, bs=32, hkv=8, d=128)
    n, hq, maxlen, part = 4, 64, 131072, 2048
    got = lib.pa_decode_workspace_bytes(n, hq, maxlen, part, ctypes.byref(d))
    cells = n * hq * (maxlen // part)
    r256 = lambda x: (x + 255) // 256 * 256
    assert got == r256(cells * 128 * 4) + r256(cells * 2 * 4)
    # one partition covers everything: no workspace
    assert lib.pa_decode_workspace_bytes(n, hq, 2048, 2048, ctypes.byref(d)) == 0


def test_auto_partition_is_block_multiple(lib):
    for bs, maxlen in ((16, 2048), (32, 131072), (16, 8192), (16, 24586)):
        d = desc(bs=bs)
        p = lib.pa_decode_partition_tokens(64, 32, maxlen, ctypes.byref(d))
        assert p > 0 and p % bs == 0
    # every kernel's sizing, including block sizes that do not divide its
    # natural unit (the CUDA-core kernel walks chunks of 8 or 16 tokens)
    for dtype in (pa.PA_BF16, pa.PA_F32):
        for dd in (40, 64, 96, 128, 200, 256):
            for bs in (1, 3, 4, 5, 8, 16, 48, 96, 128, 256):
                for hq, maxlen in ((8, 100), (32, 4096), (64, 70000)):
                    d = desc(bs=bs, d=dd, dtype=dtype)
                    p = lib.pa_decode_partition_tokens(4, hq, maxlen, ctypes.byref(d))
                    assert p > 0 and p % bs == 0, (dtype, dd, bs, hq, maxlen, p)


def test_invalid_arguments_rejected_before_any_launch(lib):
    d = desc()
    bad = pa.CacheDesc(0, 16, 8, 128, pa.PA_BF16)
    # null pointers / bad descriptors return INVALID_ARG without touching a GPU
    assert lib.pa_write_kv(None, None, None, 4, None, None, ctypes.byref(d), None) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv(None, None, None, 4, None, None, ctypes.byref(bad), None) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_write_kv(None, None, None, 0, None, None, ctypes.byref(d), None) == pa.PA_OK
    assert lib.pa_decode(None, None, None, None, 4, None, 2, 64, 32, 1.0, 0, None, None, 0,
                         ctypes.byref(d), None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(None, None, None, None, 4, None, 2, 64, 30, 1.0, 0, None, None, 0,
                         ctypes.byref(d), None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(None, None, None, None, 4, None, 0, 64, 32, 1.0, 0, None, None, 0,
                         ctypes.byref(d), None) == pa.PA_OK
    # the fused append: no new rows, or the decode's own argument errors
    assert lib.pa_decode_append(None, None, None, None, None, None, 4, None, 2, 64, 32, 1.0, 0,
                                None, None, 0, ctypes.byref(d), None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_append(None, 16, 16, None, None, None, 4, None, 2, 64, 32, 1.0, 0,
                                None, None, 0, ctypes.byref(d), None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_append(None, 16, 16, None, None, None, 4, None, 2, 64, 30, 1.0, 0,
                                None, None, 0, ctypes.byref(d), None) == pa.PA_ERR_INVALID_ARG


def test_binding_refuses_host_tensors():
    import torch
    x = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.write_kv(x, x, torch.zeros(2, dtype=torch.int64), torch.zeros(4, 8, 16, 128), x)
    c = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.decode_append(x, x, x, c, c, torch.zeros(2, 1, dtype=torch.int32),
                         torch.ones(2, dtype=torch.int32), 1)


def test_wait_check_refuses_bad_arguments_without_a_gpu(lib):
    """Argument checks run before any launch, so they need no device."""
    for args in [(0, 0, 2_000_000), (1025, 0, 2_000_000), (4, 5, 2_000_000),
                 (4, -1, 2_000_000), (4, 4, 10), (4, 4, 1 << 40)]:
        assert lib.pa_check_wait_timeout(*args, None) == pa.PA_ERR_INVALID_ARG
