// write_kv.cuh -- slot-mapping scatter of new K/V rows into the paged caches.
//
// Token j with slot s = slot_mapping[j] >= 0 lands in block s / B, row s % B
// of every kv head ("vLLM PagedAttention: from memory fragmentation to slot
// mapping" §6; paper notes' block lifecycle: decode fills the next slot of the
// last block).  A warp moves one token's rows in VEC-byte vectors; consecutive
// lanes cover one (token, head) row, then the next head, then V, so both the
// read of k/v and the write of each cache row coalesce.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace pa {

template <int VEC>
struct VecType;
template <>
struct VecType<16> { using T = uint4; };
template <>
struct VecType<8> { using T = uint2; };
template <>
struct VecType<4> { using T = uint32_t; };
template <>
struct VecType<2> { using T = uint16_t; };

// Slot of token j from a precomputed slot mapping (s < 0: skip).
struct SlotFromMapping {
    const int64_t* slot_mapping;
    __device__ __forceinline__ int64_t operator()(int64_t j, bool /*report*/) const {
        return __ldg(slot_mapping + j);
    }
};

// Slot of token j computed on the device from its sequence and position:
// table[seq][pos / B] * B + pos % B ("vLLM PagedAttention: from memory
// fragmentation to slot mapping" §3 formula; §6: positions plus the device
// block table give the slot mapping).  A negative sequence id or position
// means "skip"; a sequence, position or table entry outside the table or the
// pool is skipped and reported.
struct SlotFromPosition {
    const int32_t* seq_ids;
    const int32_t* positions;
    const int32_t* block_tables;
    int32_t num_seqs, max_blocks, block_size, num_blocks;
    __device__ __forceinline__ int64_t operator()(int64_t j, bool report) const {
        const int32_t s = __ldg(seq_ids + j), p = __ldg(positions + j);
        if (s < 0 || p < 0) return -1;
        if (s >= num_seqs || (int64_t)p >= (int64_t)max_blocks * block_size) {
            if (report) raise_error(PA_DEVERR_TABLE_ENTRY);
            return -1;
        }
        const int32_t id = __ldg(block_tables + (int64_t)s * max_blocks + p / block_size);
        if (id < 0 || id >= num_blocks) {
            if (report) raise_error(PA_DEVERR_TABLE_ENTRY);
            return -1;
        }
        return (int64_t)id * block_size + p % block_size;
    }
};

// Slot of sequence j's newest token in a decode step: position
// seq_lens[j] - 1 (lengths count the new token; paper notes' block
// lifecycle: decode fills the next slot of the last block), through the same
// table formula.  A length of 0 appends nothing; a length the table or the
// host bound cannot hold (reported as the decode reports it), or a bad table
// entry, is skipped and reported.
struct SlotFromAppend {
    const int32_t* seq_lens;
    const int32_t* block_tables;
    int32_t max_blocks, block_size, num_blocks, max_seq_len;
    __device__ __forceinline__ int64_t operator()(int64_t j, bool report) const {
        const int32_t t = __ldg(seq_lens + j);
        if (t == 0) return -1;
        const int64_t cap = min((int64_t)max_seq_len, (int64_t)max_blocks * block_size);
        if (t < 0 || t > cap) {
            if (report) raise_error(PA_DEVERR_SEQ_LEN);
            return -1;
        }
        const int32_t p = t - 1;
        const int32_t id = __ldg(block_tables + j * max_blocks + p / block_size);
        if (id < 0 || id >= num_blocks) {
            if (report) raise_error(PA_DEVERR_TABLE_ENTRY);
            return -1;
        }
        return (int64_t)id * block_size + p % block_size;
    }
};

// One warp per token (a grid-stride loop over tokens): every lane reads the
// token's slot (one broadcast load), then the warp moves the token's
// 2 * Hkv * row_bytes bytes, each lane issuing up to kWriteUnroll vector
// loads before its stores, so a warp keeps 32 * kWriteUnroll vectors in
// flight.  Vector x of a token is (K or V, head, piece): K rows first, head
// by head, so consecutive lanes read and write consecutive bytes.
constexpr int kWriteUnroll = 8;
constexpr int kWriteWarps = 8;                  // warps per CTA

template <int VEC, typename SlotFn>
__global__ void __launch_bounds__(32 * kWriteWarps, 2)
write_kv_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v, SlotFn slot_of,
                int64_t num_tokens, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                int32_t num_kv_heads, int32_t block_size, int64_t num_slots,
                int32_t row_bytes) {
    using V = typename VecType<VEC>::T;
    griddep_wait();                 // inputs may come from the previous kernel
    griddep_launch_dependents();    // the next kernel may start its prologue
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t vpr = row_bytes / VEC;                  // vectors per (token, head) row
    const int32_t per_kind = num_kv_heads * vpr;           // vectors of K (or V) of a token
    const int32_t per_token = 2 * per_kind;
    for (int64_t j = (int64_t)blockIdx.x * kWriteWarps + warp; j < num_tokens;
         j += (int64_t)gridDim.x * kWriteWarps) {
        const int64_t s = slot_of(j, lane == 0);          // one report per token
        if (s < 0) continue;
        if (s >= num_slots) {
            if (lane == 0) raise_error(PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = s / block_size;
        const int64_t row = s - blk * block_size;
        const int64_t src0 = j * num_kv_heads * (int64_t)row_bytes;
        // cache row of head h: ((blk * Hkv + h) * B + row) * row_bytes
        const int64_t dst0 = (blk * num_kv_heads * block_size + row) * (int64_t)row_bytes;
        const int64_t head_stride = (int64_t)block_size * row_bytes;
        for (int32_t x0 = 0; x0 < per_token; x0 += 32 * kWriteUnroll) {
            V buf[kWriteUnroll];
#pragma unroll
            for (int u = 0; u < kWriteUnroll; ++u) {
                const int32_t x = x0 + u * 32 + lane;
                if (x < per_token) {
                    const int32_t which = x >= per_kind;      // 0 = K, 1 = V
                    const int32_t y = x - which * per_kind;   // head * vpr + piece
                    buf[u] = *reinterpret_cast<const V*>((which ? v : k) + src0 +
                                                         (int64_t)y * VEC);
                }
            }
#pragma unroll
            for (int u = 0; u < kWriteUnroll; ++u) {
                const int32_t x = x0 + u * 32 + lane;
                if (x < per_token) {
                    const int32_t which = x >= per_kind;
                    const int32_t y = x - which * per_kind;
                    const int32_t h = y / vpr, c = y - h * vpr;
                    *reinterpret_cast<V*>((which ? v_cache : k_cache) + dst0 +
                                          h * head_stride + (int64_t)c * VEC) = buf[u];
                }
            }
        }
    }
}

// Whole-block copies for copy-on-write and swapping: for each pair (src, dst)
// every byte of block src of the source K and V caches goes to block dst of
// the destination caches (nxmr.cn article §4.2: copy the old block's K/V into
// the new one; paper notes: swapping moves a preempted sequence's blocks
// between GPU and CPU memory).  Either side may be page-locked host memory.
// Consecutive threads move consecutive 16-byte pieces of one block.
template <int VEC>
__global__ void __launch_bounds__(256)
copy_blocks_kernel(const uint8_t* __restrict__ src_k, const uint8_t* __restrict__ src_v,
                   int64_t src_blocks, uint8_t* __restrict__ dst_k, uint8_t* __restrict__ dst_v,
                   int64_t dst_blocks, const int64_t* __restrict__ pairs, int64_t num_pairs,
                   int64_t block_bytes) {
    using V = typename VecType<VEC>::T;
    griddep_wait();
    griddep_launch_dependents();
    const int64_t vecs = block_bytes / VEC;
    const int64_t per_pair = 2 * vecs;
    const int64_t total = num_pairs * per_pair;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = idx / per_pair;
        int64_t c = idx - j * per_pair;
        const int which = c >= vecs;
        c -= which * vecs;
        const int64_t s = pairs[2 * j], d = pairs[2 * j + 1];
        if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
            if (which == 0 && c == 0) raise_error(PA_DEVERR_BLOCK_PAIR);
            continue;
        }
        const uint8_t* from = (which ? src_v : src_k) + s * block_bytes + c * VEC;
        uint8_t* to = (which ? dst_v : dst_k) + d * block_bytes + c * VEC;
        *reinterpret_cast<V*>(to) = *reinterpret_cast<const V*>(from);
    }
}

}  // namespace pa
