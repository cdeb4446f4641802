// merge.cuh -- log-sum-exp merge of split-K partitions.
//
// For a sequence split into n > 1 partitions, each (sequence, query head) has
// per-partition (acc_p, m_p, l_p) in the workspace (m in base-2 units).  With
// M = max_p m_p and w_p = 2^(m_p - M):
//     out = sum_p w_p acc_p / sum_p w_p l_p
// (the V2 kernel's reduce step in "vLLM source walkthrough: PagedAttention and
// Continuous Batching" §1.8; one global softmax over all blocks' raw scores,
// paper notes' 10-token example).
//
// One CTA per (sequence, query head).  Up to kMergeSmall partitions, each
// thread loads every (m_p, l_p) and its own columns of acc_p in one go and
// reduces them in partition order.  Beyond that the CTA reduces M and L over
// the partitions, stages the weights w_p in shared memory one tile at a time,
// and each thread accumulates its output columns over the partitions, so the
// partial reads are coalesced across threads and independent across
// partitions.  Every reduction has a fixed order: the result is deterministic.
#pragma once

#include "decode_generic.cuh"

namespace pa {

constexpr int kMergeThreads = 128;
constexpr int kMergeTile = 512;    // partition weights staged per pass
constexpr int kMergeSmall = 16;    // up to this many partitions: one-pass path

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();                       // red[] free from any earlier use
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

template <typename E>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeArgs a) {
    __shared__ float w_sm[kMergeTile];
    __shared__ float red[kMergeThreads / 32];
    griddep_wait();                                   // partials of the decode kernel
    const int64_t pair = blockIdx.x;                  // sequence * Hq + head
    const int32_t i = (int32_t)(pair / a.num_q_heads);
    const int32_t T = checked_len(a, i);
    const int32_t n = (int32_t)(((int64_t)T + a.part_tokens - 1) / a.part_tokens);
    if (n <= 1) return;   // written directly by the partition kernel
    const int32_t tid = threadIdx.x;
    const int64_t cell0 = pair * a.max_parts;
    const float* ml = a.ws_ml + 2 * cell0;
    const float* acc = a.ws_acc + cell0 * a.head_dim;
    E* out = static_cast<E*>(a.out) + pair * a.head_dim;

    if (n <= kMergeSmall) {
        // few partitions: every thread loads all (m, l) and its columns' acc
        // at once (one memory round trip), then reduces them in order
        for (int32_t d0 = 0; d0 < a.head_dim; d0 += kMergeThreads) {
            const int32_t d = d0 + tid;
            float mv[kMergeSmall], lv[kMergeSmall], av[kMergeSmall];
#pragma unroll
            for (int p = 0; p < kMergeSmall; ++p) {
                if (p < n) {
                    mv[p] = ml[2 * p];
                    lv[p] = ml[2 * p + 1];
                    av[p] = d < a.head_dim ? acc[(int64_t)p * a.head_dim + d] : 0.f;
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int p = 0; p < kMergeSmall; ++p)
                if (p < n) M = fmaxf(M, mv[p]);
            float L = 0.f, A = 0.f;
#pragma unroll
            for (int p = 0; p < kMergeSmall; ++p) {
                if (p < n && mv[p] != -INFINITY) {
                    const float w = exp2f(mv[p] - M);
                    L += w * lv[p];
                    A += w * av[p];
                }
            }
            if (d < a.head_dim) out[d] = Elem<E>::from_float(L > 0.f ? A / L : 0.f);
        }
        return;
    }

    float m = -INFINITY;
    for (int32_t p = tid; p < n; p += kMergeThreads) m = fmaxf(m, ml[2 * p]);
    const float M = block_reduce(m, true, red);
    float l = 0.f;
    for (int32_t p = tid; p < n; p += kMergeThreads) {
        const float mp = ml[2 * p];
        if (mp != -INFINITY) l += exp2f(mp - M) * ml[2 * p + 1];
    }
    const float L = block_reduce(l, false, red);
    const float inv = L > 0.f ? 1.f / L : 0.f;

    // columns in groups of 2 * kMergeThreads: each thread owns two of them
    for (int32_t d0 = 0; d0 < a.head_dim; d0 += 2 * kMergeThreads) {
        float o[2] = {0.f, 0.f};
        for (int32_t p0 = 0; p0 < n; p0 += kMergeTile) {
            const int32_t cnt = min(kMergeTile, n - p0);
            __syncthreads();
            for (int32_t p = tid; p < cnt; p += kMergeThreads) {
                const float mp = ml[2 * (p0 + p)];
                w_sm[p] = mp == -INFINITY ? 0.f : exp2f(mp - M);
            }
            __syncthreads();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int32_t d = d0 + tid + c * kMergeThreads;
                if (d < a.head_dim) {
                    float s = 0.f;
#pragma unroll 32
                    for (int32_t p = 0; p < cnt; ++p)
                        s += w_sm[p] * acc[(int64_t)(p0 + p) * a.head_dim + d];
                    o[c] += s;
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int32_t d = d0 + tid + c * kMergeThreads;
            if (d < a.head_dim) out[d] = Elem<E>::from_float(o[c] * inv);
        }
    }
}

}  // namespace pa
