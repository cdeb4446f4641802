"""The bounded pipeline wait on a live GPU: a barrier left short of its
arrivals makes the wait give up after its bound.  The bit PA_DEVERR_TIMEOUT
is raised, nothing faults, and the context stays usable: a decode right
after matches the oracle.  Nothing here can hang: every wait has a bound of
a few million clocks (about a millisecond)."""
import time

import pytest
import torch

import paged_kv_cache_109_gb300 as pa
from paged_kv_cache_109_gb300 import workloads
from tests._gpu import BF16_ATOL, BF16_RTOL, DeviceState, HostState, assert_close

pytestmark = pytest.mark.gpu

LIMIT = 2_000_000          # SM clocks: about 1 ms at 2 GHz


@pytest.fixture(autouse=True)
def clear_device_error(cuda_device):
    pa.last_device_error()
    yield


@pytest.mark.parametrize("expected", [1, 32, 64, 1000])
def test_completed_phase_raises_nothing(cuda_device, expected):
    pa.check_wait_timeout(expected, expected, LIMIT)
    assert pa.last_device_error() == 0


@pytest.mark.parametrize("expected, arrivals", [(1, 0), (64, 63), (1000, 1)])
def test_wait_short_of_arrivals_times_out_and_reports(cuda_device, expected, arrivals):
    t0 = time.perf_counter()
    pa.check_wait_timeout(expected, arrivals, LIMIT)
    bits = pa.last_device_error()                  # synchronises
    elapsed = time.perf_counter() - t0
    assert bits == pa.DEVERR_TIMEOUT
    assert elapsed < 5.0                           # the bound ended the wait
    assert pa.last_device_error() == 0             # read once, then cleared


def test_context_stays_usable_after_a_timeout(cuda_device):
    pa.check_wait_timeout(32, 0, LIMIT)
    assert pa.last_device_error() == pa.DEVERR_TIMEOUT
    wl = workloads.make("gqa", num_seqs=8, median_len=300, max_len=2000, num_shared=2,
                        prefix_len=128, num_blocks=1024)
    st = wl.steps[0]
    d, h = DeviceState(wl, cuda_device), HostState(wl)
    d.write(st)
    h.write(st)
    out = d.decode(st)
    torch.cuda.synchronize()
    assert pa.last_device_error() == 0
    assert_close(out.cpu().double().numpy(), h.decode(st), BF16_ATOL, BF16_RTOL, "decode")


def test_bad_arguments_are_refused_before_launch(cuda_device):
    lib = pa.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for args in [(0, 0, LIMIT), (1025, 0, LIMIT), (4, 5, LIMIT), (4, -1, LIMIT),
                 (4, 4, 10), (4, 4, 1 << 40)]:
        assert lib.pa_check_wait_timeout(*args, stream) == pa.PA_ERR_INVALID_ARG
    assert pa.last_device_error() == 0
