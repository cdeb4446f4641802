// decode_config.cuh -- decode tuning knobs, kernel selection and split-K
// sizing (host side).  The automatic partition size decides how many CTAs a
// call launches and how many split partials it writes, so it belongs with
// the kernels it configures.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "decode_tiled.cuh"
#include "pa.h"

#ifndef PA_USE_PDL
#define PA_USE_PDL 1   // launch with programmatic stream serialization
#endif
#ifndef PA_TARGET_CTAS_PER_SM
#define PA_TARGET_CTAS_PER_SM 8
#endif
#ifndef PA_MAX_PARTITION_TOKENS
#define PA_MAX_PARTITION_TOKENS 1024
#endif
#ifndef PA_LONG_PARTITIONS
#define PA_LONG_PARTITIONS 32   // TMA kernel: the cap rises to max_seq_len / this
#endif

namespace pa {
namespace {

constexpr int kMaxDevices = 64;

int device_sm_count() {
    static int cached[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

// ---- kernel selection --------------------------------------------------------

// Groups of more than 16 query heads are split into sub-groups of 16, one CTA
// each, reading the same K/V tiles (the later reads mostly hit L2).  Every
// head dim that is a multiple of 16 up to 128 loads as 64-column boxes (one
// up to 64, two above) whose columns past the head dim are zero-filled by
// the copy (out of the tensor map's bounds) and never read from memory.
// Head dim 256 (four boxes) runs at one CTA per SM for groups of two or
// more query heads; a single head per kv head stays on the tiled kernel,
// measured a little faster there (0.88 against 0.86 of the copy peak).
bool tma_head_dim(int32_t D, int32_t group) {
    return (D % 16 == 0 && D >= 16 && D <= 128) || (D == 256 && group >= 2);
}

bool fast_shape(const pa_cache_desc* c, int32_t group) {
    if (c->dtype != PA_BF16 || group < 1) return false;
    const int D = c->head_dim, B = c->block_size;
    if (!tma_head_dim(D, group)) return false;
    return B == 8 || (B % 16 == 0 && B <= 256);
}

// The tiled CUDA-core kernel: head dims up to 256 whose rows are whole
// 16-byte pieces (its copies are 16 bytes; the caches must be 16-byte aligned,
// which the caller checks).
bool tiled_shape(const pa_cache_desc* c) {
    const int e = c->dtype == PA_F32 ? 4 : 2;
    return c->head_dim <= 256 && (c->head_dim * e) % 16 == 0;
}

#ifndef PA_DECODE_MMA_MIN_GROUP
#define PA_DECODE_MMA_MIN_GROUP 5
#endif

// The mma.sync kernel: bf16 head dims that are multiples of 16 up to 128 the
// TMA kernel does not take (16, 32, 48, and every head dim at block sizes
// other than 8 or a multiple of 16), for groups of at least
// PA_DECODE_MMA_MIN_GROUP query heads.  Smaller groups stay on the tiled
// CUDA-core kernel: its run copies move a block's rows with one copy each,
// where this kernel copies every row on its own (to pad it), and at up to
// four heads the CUDA cores keep up with HBM.  Measured, fraction of the copy
// peak (tiled / mma.sync), before head dims 80-112 moved to the TMA kernel:
// G = 1, D = 96: 0.886 / 0.467; G = 4, D = 96: 0.487 / 0.452; G = 4, B = 4:
// 0.615 / 0.582; G = 8, D = 64, B = 4: 0.210 / 0.374; G = 16, D = 112:
// 0.169 / 0.433.
bool mma_shape(const pa_cache_desc* c, int32_t group) {
    return c->dtype == PA_BF16 && c->head_dim % 16 == 0 && c->head_dim <= 128 &&
           group >= PA_DECODE_MMA_MIN_GROUP && !fast_shape(c, group);
}

// Largest partition (tokens) the generic kernel's shared memory holds.
int32_t generic_max_partition(const pa_cache_desc* c, int32_t group) {
    const size_t budget = 96 * 1024;
    int32_t B = c->block_size;
    int64_t fixed = 4LL * ((int64_t)group * c->head_dim + 2 * group);
    int64_t per_tok = 4LL * group;
    int64_t p = (int64_t(budget) - fixed) / per_tok;
    p = p / B * B;
    return (int32_t)std::max<int64_t>(p, 0);
}

int32_t fast_max_partition(const pa_cache_desc* c) {
    return 2048 * c->block_size;   // TmaMmaCfg::kMaxTableSlice blocks
}

int32_t auto_partition(int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                       const pa_cache_desc* c) {
    const int32_t B = c->block_size;
    const int32_t group = num_q_heads / c->num_kv_heads;
    const bool fast = fast_shape(c, group);
    const bool mma = mma_shape(c, group);
    if (!fast && !mma && !tiled_shape(c)) {
        int32_t cap = generic_max_partition(c, group);
        int32_t want = std::max(B, (512 / B) * B);
        return std::max(B, std::min(cap, want));
    }
    // TMA kernel: one block per warp per step; mma.sync and tiled kernels: a
    // chunk for each of their four warps, rounded up to whole blocks.  Aim for about
    // PA_TARGET_CTAS_PER_SM CTAs per SM over the batch (counted at
    // max_seq_len, sub-groups included), between one unit and
    // PA_MAX_PARTITION_TOKENS tokens.  On the TMA kernel the cap rises to
    // max_seq_len / PA_LONG_PARTITIONS for sequences long enough that it
    // binds: there the batch's CTA count never runs short, and fewer, longer
    // partitions cost fewer partials to write and merge.  Measured on the
    // long-context batch (4 x 131072, Hkv = 8, 1216 CTAs at the target): 1024
    // tokens 1.034-1.037 of the copy peak per call, 2048 1.057, 3456 (the
    // target) 1.070; the batches whose longest sequence is under 32768 tokens
    // keep 1024, which measured best or within 1% for them.
    const int64_t chunks = mma ? 4 * 16
                               : (int64_t)kTiledWarps *
                                     tiled_chunk(c->head_dim, c->dtype == PA_F32 ? 4 : 2);
    const int64_t unit = fast ? 4LL * B : (chunks + B - 1) / B * B;   // whole blocks
    const int64_t sms = std::max(1, device_sm_count());
    const int64_t heads_per_cta = fast || mma ? 16 : 8;
    const int64_t work = (int64_t)num_seqs * c->num_kv_heads *
                         ((group + heads_per_cta - 1) / heads_per_cta) *
                         std::max(max_seq_len, 1);
    const int64_t target = (int64_t)PA_TARGET_CTAS_PER_SM * sms;
    int64_t p = (work + target - 1) / target;
    p = (p + unit - 1) / unit * unit;
    int64_t cap = std::max<int64_t>(unit, PA_MAX_PARTITION_TOKENS / unit * unit);
    if (fast) cap = std::max<int64_t>(cap, (int64_t)max_seq_len / PA_LONG_PARTITIONS / unit * unit);
    p = std::min(std::max(p, unit), cap);
    if (fast) p = std::min<int64_t>(p, fast_max_partition(c));
    return (int32_t)p;
}

// Partitions of the longest sequence, in 64-bit arithmetic (max_seq_len + part
// overflows int32 near INT32_MAX).  The launch refuses more than 65535.
int64_t num_parts(int32_t max_seq_len, int32_t part) {
    return std::max<int64_t>(1, ((int64_t)max_seq_len + part - 1) / part);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                       int32_t part, const pa_cache_desc* c) {
    const int64_t P = num_parts(max_seq_len, part);
    if (P <= 1) return 0;
    const size_t cells = (size_t)num_seqs * num_q_heads * P;
    return align256(cells * c->head_dim * sizeof(float)) + align256(cells * 2 * sizeof(float));
}

}  // namespace
}  // namespace pa
