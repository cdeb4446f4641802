// write_kv.cuh -- slot-mapping scatter of new K/V rows into the paged caches.
//
// Token j with slot s = slot_mapping[j] >= 0 lands in block s / B, row s % B
// of every kv head ("vLLM PagedAttention: from memory fragmentation to slot
// mapping" §6; paper notes' block lifecycle: decode fills the next slot of the
// last block).  Each thread moves one VEC-byte vector; consecutive threads
// cover one (token, head) row, then the next head, then V, then the next
// token, so both the read of k/v and the write of each cache row coalesce.
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

template <int VEC, typename SlotFn>
__global__ void __launch_bounds__(256)
write_kv_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v, SlotFn slot_of,
                int64_t num_tokens, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                int32_t num_kv_heads, int32_t block_size, int64_t num_slots,
                int32_t row_bytes) {
    using V = typename VecType<VEC>::T;
    griddep_wait();                 // inputs may come from the previous kernel
    griddep_launch_dependents();    // the next kernel may start its prologue
    const int64_t vecs_per_row = row_bytes / VEC;
    const int64_t per_token = 2LL * num_kv_heads * vecs_per_row;
    const int64_t total = num_tokens * per_token;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = idx / per_token;
        int64_t rem = idx - j * per_token;
        const int which = rem >= num_kv_heads * vecs_per_row;   // 0 = K, 1 = V
        rem -= which * num_kv_heads * vecs_per_row;
        const int64_t h = rem / vecs_per_row;
        const int64_t c = rem - h * vecs_per_row;
        const bool first = which == 0 && h == 0 && c == 0;    // one report per token
        const int64_t s = slot_of(j, first);
        if (s < 0) continue;
        if (s >= num_slots) {
            if (first) raise_error(PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = s / block_size;
        const int64_t row = s - blk * block_size;
        const uint8_t* src = (which ? v : k) + (j * num_kv_heads + h) * row_bytes + c * VEC;
        uint8_t* dst = (which ? v_cache : k_cache) +
                       ((blk * num_kv_heads + h) * block_size + row) * row_bytes + c * VEC;
        *reinterpret_cast<V*>(dst) = *reinterpret_cast<const V*>(src);
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
