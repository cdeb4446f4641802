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

template <int VEC>
__global__ void __launch_bounds__(256)
write_kv_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
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
        const int64_t s = __ldg(slot_mapping + j);
        if (s < 0) continue;
        if (s >= num_slots) {
            if (which == 0 && h == 0 && c == 0) raise_error(PA_DEVERR_SLOT);
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

}  // namespace pa
