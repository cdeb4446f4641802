"""Helpers shared by the GPU parity tests: run one workload step through the C
ABI and through the CPU oracle, and compare."""
import numpy as np
import torch

import oracle
import paged_kv_cache_109_gb300 as pa

BF16_ATOL, BF16_RTOL = 3e-3, 1e-2     # bf16 path vs fp64 oracle on the same bf16 inputs
F32_ATOL = 1e-5                        # fp32 path: max abs error


def assert_close(got, ref, atol, rtol, what="", extra=None):
    """|got - ref| <= atol + rtol |ref| (+ extra, per element, where given)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    if extra is not None:
        bound = bound + np.asarray(extra, dtype=np.float64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} beyond atol={atol} "
                             f"rtol={rtol}; max abs err {float(np.nanmax(err)):.3e}; first {idx}")


def tolerance(dtype):
    return (F32_ATOL, 0.0) if dtype == torch.float32 else (BF16_ATOL, BF16_RTOL)


class DeviceState:
    """Device copies of a workload's caches, advanced step by step."""

    def __init__(self, wl, dev):
        self.wl = wl
        self.dev = dev
        self.k_cache = wl.k_cache.to(dev)
        self.v_cache = wl.v_cache.to(dev)

    def write(self, step):
        pa.write_kv(step.k_new.to(self.dev), step.v_new.to(self.dev),
                    step.slot_mapping.to(self.dev), self.k_cache, self.v_cache)

    def decode(self, step, **kw):
        return pa.decode(step.q.to(self.dev), self.k_cache, self.v_cache,
                         step.block_tables.to(self.dev), step.seq_lens.to(self.dev),
                         int(step.seq_lens.max()), self.wl.scale, **kw)


    def append(self, step, **kw):
        """The step's write and decode in one pa_decode_append call (steps
        whose new tokens are each sequence's last position)."""
        return pa.decode_append(step.q.to(self.dev), step.k_new.to(self.dev),
                                step.v_new.to(self.dev), self.k_cache, self.v_cache,
                                step.block_tables.to(self.dev), step.seq_lens.to(self.dev),
                                int(step.seq_lens.max()), self.wl.scale, **kw)


class HostState:
    """Oracle-side copies of the caches, advanced with the oracle's write."""

    def __init__(self, wl):
        self.wl = wl
        self.k_cache = wl.k_cache.clone()
        self.v_cache = wl.v_cache.clone()

    def write(self, step):
        assert oracle.write_kv(step.k_new, step.v_new, step.slot_mapping, self.k_cache,
                               self.v_cache) == 0

    def decode(self, step, pairs=None):
        return oracle.decode(step.q, self.k_cache, self.v_cache, step.block_tables,
                             step.seq_lens, self.wl.scale, pairs=pairs)


def sample_pairs(step, num_q_heads, count, seed=0):
    """(seq, head) pairs: every head of the longest and shortest sequence plus
    `count` seeded random ones."""
    rng = np.random.default_rng(seed)
    lens = step.seq_lens.numpy()
    n = lens.shape[0]
    pairs = {(int(lens.argmax()), h) for h in range(num_q_heads)}
    pairs |= {(int(lens.argmin()), h) for h in range(num_q_heads)}
    for _ in range(count):
        pairs.add((int(rng.integers(n)), int(rng.integers(num_q_heads))))
    return np.array(sorted(pairs), dtype=np.int64)


def decode_kernel(dtype, d, bs, group):
    """The decode kernel pa_decode_path names for a shape: 1 TMA + tensor
    cores (bf16 head dims that are multiples of 16 up to 128, and 256 with
    groups of two or more, at block sizes 8 and multiples of 16), 2 mma.sync
    (groups of 5 or more heads on the head dims up to 128 at other block
    sizes), 0 CUDA cores (fp32 and the rest)."""
    tma_d = (d % 16 == 0 and 16 <= d <= 128) or (d == 256 and group >= 2)
    if dtype == torch.bfloat16 and tma_d and (bs == 8 or (bs % 16 == 0 and bs <= 256)):
        return 1
    if dtype == torch.bfloat16 and d % 16 == 0 and d <= 128 and group >= 5:
        return 2
    return 0
