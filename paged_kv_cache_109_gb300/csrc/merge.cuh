// merge.cuh -- log-sum-exp merge of split-K partitions.
//
// For a sequence split into n > 1 partitions, each (sequence, query head) has
// per-partition (acc_p, m_p, l_p) in the workspace (m in base-2 units).  With
// M = max_p m_p and w_p = 2^(m_p - M):
//     out = sum_p w_p acc_p / sum_p w_p l_p
// (the V2 kernel's reduce step in "vLLM source walkthrough: PagedAttention and
// Continuous Batching" §1.8; one global softmax over all blocks' raw scores,
// paper notes' 10-token example).  One warp per (sequence, head); partitions
// are combined in index order, so the result is deterministic.
#pragma once

#include "decode_generic.cuh"

namespace pa {

template <typename E>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeArgs a) {
    const int32_t warps = blockDim.x / 32;
    const int64_t pair = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    const int32_t lane = threadIdx.x & 31;
    const int64_t num_pairs = (int64_t)a.num_seqs * a.num_q_heads;
    if (pair >= num_pairs) return;
    const int32_t i = (int32_t)(pair / a.num_q_heads);
    const int32_t T = checked_len(a, i);
    const int32_t n = (T + a.part_tokens - 1) / a.part_tokens;
    if (n <= 1) return;   // written directly by the partition kernel
    const int64_t cell0 = pair * a.max_parts;
    float M = -INFINITY;
    for (int32_t p = 0; p < n; ++p) M = fmaxf(M, a.ws_ml[2 * (cell0 + p)]);
    float L = 0.f;
    for (int32_t p = 0; p < n; ++p) {
        const float m = a.ws_ml[2 * (cell0 + p)];
        L += (m == -INFINITY ? 0.f : exp2f(m - M)) * a.ws_ml[2 * (cell0 + p) + 1];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    E* out = static_cast<E*>(a.out) + pair * a.head_dim;
    for (int32_t d = lane; d < a.head_dim; d += 32) {
        float acc = 0.f;
        for (int32_t p = 0; p < n; ++p) {
            const float m = a.ws_ml[2 * (cell0 + p)];
            if (m != -INFINITY) acc += exp2f(m - M) * a.ws_acc[(cell0 + p) * a.head_dim + d];
        }
        out[d] = Elem<E>::from_float(acc * inv);
    }
}

}  // namespace pa
