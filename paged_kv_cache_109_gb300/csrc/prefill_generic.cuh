// prefill_generic.cuh -- portable multi-query (chunked prefill) attention for
// fp32 caches and shapes the TMA + tensor-core kernel does not cover.
//
// One CTA per (query row r, kv head g); warp w takes query heads g*G + w,
// g*G + w + 4, ...; lanes split the head dimension.  The row's sequence i is
// found by binary search in query_start; its position is
// p = T_i - L_i + (r - query_start[i]) and it attends to keys 0..p with an
// online softmax (the same definition as the TMA kernel and the oracle).
#pragma once

#include "prefill_args.cuh"

namespace pa {

constexpr int kGenericMaxDimPerLane = 8;   // head_dim <= 256

template <typename E>
__global__ void __launch_bounds__(128) prefill_generic_kernel(const PrefillArgs a) {
    griddep_wait();
    const int32_t r = blockIdx.x, g = blockIdx.y;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t D = a.head_dim, G = a.group, BS = a.block_size;
    // sequence of row r: the last i with query_start[i] <= r
    int32_t lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) / 2;
        if (a.query_start[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int32_t i = lo;
    const int32_t q0 = a.query_start[i], L = a.query_start[i + 1] - q0;
    const int32_t T = clamp_len(a, a.seq_lens[i]);
    if (L > T || r - q0 >= L) {
        if (threadIdx.x == 0 && g == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int32_t p = T - L + (r - q0);
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;
    const E* q = static_cast<const E*>(a.q);
    const E* kc = static_cast<const E*>(a.k_cache);
    const E* vc = static_cast<const E*>(a.v_cache);
    E* out = static_cast<E*>(a.out);
    for (int32_t hh = warp; hh < G; hh += blockDim.x / 32) {
        const int32_t h = g * G + hh;
        float qv[kGenericMaxDimPerLane], acc[kGenericMaxDimPerLane];
#pragma unroll
        for (int j = 0; j < kGenericMaxDimPerLane; ++j) {
            const int32_t d = lane + 32 * j;
            qv[j] = d < D ? Elem<E>::to_float(q[((int64_t)r * a.num_q_heads + h) * D + d]) : 0.f;
            acc[j] = 0.f;
        }
        float m = -INFINITY, l = 0.f;
        for (int32_t t = 0; t <= p; ++t) {
            const int32_t id = table[t / BS];
            if (id < 0 || id >= a.num_blocks) {
                if (lane == 0) raise_error(PA_DEVERR_TABLE_ENTRY);
                continue;
            }
            const int64_t row = (((int64_t)id * a.num_kv_heads + g) * BS + t % BS) * D;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < kGenericMaxDimPerLane; ++j) {
                const int32_t d = lane + 32 * j;
                if (d < D) dot += qv[j] * Elem<E>::to_float(kc[row + d]);
            }
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float sc = dot * a.scale_log2;
            const float mn = fmaxf(m, sc);
            const float al = exp2f(m - mn), w = exp2f(sc - mn);
            m = mn;
            l = l * al + w;
#pragma unroll
            for (int j = 0; j < kGenericMaxDimPerLane; ++j) {
                const int32_t d = lane + 32 * j;
                if (d < D) acc[j] = acc[j] * al + w * Elem<E>::to_float(vc[row + d]);
            }
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int j = 0; j < kGenericMaxDimPerLane; ++j) {
            const int32_t d = lane + 32 * j;
            if (d < D) out[((int64_t)r * a.num_q_heads + h) * D + d] = Elem<E>::from_float(acc[j] * inv);
        }
    }
}

}  // namespace pa
