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
// One CTA of W warps per (sequence, query head).  Warp w owns partitions
// w, w + W, w + 2W, ...; each lane owns VEC consecutive columns of a 32 * VEC
// column slab (float4 loads when the head dim is a multiple of 4).  A warp
// issues the loads of kMergeChunk of its partitions at once (one memory round
// trip for up to W * kMergeChunk partitions), takes their maximum, rescales
// its running (m, l, acc) to it and adds the chunk.  The W running states are
// then combined through shared memory in warp order.  Every step has a fixed
// order for a given n and W, so the result is deterministic.
//
// The chunk is 4 partitions deep (40-62 registers).  Measured on the GQA and
// continuous-batching batches (thousands of (sequence, head) pairs with a few
// partitions each), 8- and 16-deep chunks take 70-160 registers, fewer merge
// CTAs fit on an SM, and the decode call is 1.5-2.5% slower; on the
// long-context batch (128 partitions per pair) the depth makes no difference.
#pragma once

#include "decode_generic.cuh"

namespace pa {

#ifndef PA_MERGE_CHUNK
#define PA_MERGE_CHUNK 4
#endif
constexpr int kMergeChunk = PA_MERGE_CHUNK;   // partitions whose loads a warp has in flight at once

template <int VEC>
struct MergeVec;
template <>
struct MergeVec<4> {
    using T = float4;
    static __device__ __forceinline__ void get(const T& v, float* x) {
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
};
template <>
struct MergeVec<1> {
    using T = float;
    static __device__ __forceinline__ void get(const T& v, float* x) { x[0] = v; }
};

// Running state of one warp: (m, l) shared by its lanes, acc per lane column.
template <int VEC>
__device__ __forceinline__ void merge_chunk(const float* __restrict__ ml,
                                            const float* __restrict__ acc, int32_t D,
                                            int32_t col, bool col_ok, int32_t p0, int32_t stride,
                                            int32_t n, float& m, float& l, float (&o)[VEC]) {
    using V = typename MergeVec<VEC>::T;
    float mp[kMergeChunk], lp[kMergeChunk];
    V ap[kMergeChunk];
    // all loads first: one round trip for the chunk
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
        const int32_t p = p0 + j * stride;
        mp[j] = -INFINITY;
        lp[j] = 0.f;
        ap[j] = V{};
        if (p < n) {
            const float2 v = *reinterpret_cast<const float2*>(ml + 2 * (int64_t)p);
            mp[j] = v.x;
            lp[j] = v.y;
            if (col_ok) ap[j] = *reinterpret_cast<const V*>(acc + (int64_t)p * D + col);
        }
    }
    float mc = m;
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) mc = fmaxf(mc, mp[j]);
    if (mc == -INFINITY) return;                 // nothing in this chunk or before
    const float r = m == -INFINITY ? 0.f : exp2f(m - mc);
    l *= r;
#pragma unroll
    for (int c = 0; c < VEC; ++c) o[c] *= r;
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
        if (mp[j] != -INFINITY) {
            const float w = exp2f(mp[j] - mc);
            float x[VEC];
            MergeVec<VEC>::get(ap[j], x);
            l += w * lp[j];
#pragma unroll
            for (int c = 0; c < VEC; ++c) o[c] += w * x[c];
        }
    }
    m = mc;
}

template <typename E, int W, int VEC>
__global__ void __launch_bounds__(32 * W) merge_kernel(const DecodeArgs a) {
    constexpr int kSlab = 32 * VEC;              // columns per pass
    __shared__ float m_sm[W], l_sm[W];
    __shared__ __align__(16) float o_sm[W][kSlab];
    griddep_wait();                              // partials of the decode kernel
    const int64_t pair = blockIdx.x;             // sequence * Hq + head
    const int32_t i = (int32_t)(pair / a.num_q_heads);
    const int32_t T = checked_len(a, i);
    int32_t n = (int32_t)(((int64_t)T + a.part_tokens - 1) / a.part_tokens);
    const int32_t k = seq_group_of(a, i);       // -1 outside a shared-prefix call
    if (k >= 0) {
        // a group member: its group's prefix partitions (slots 0 ..), then its
        // own past the shared blocks; merged even when there is one (its
        // partials are not normalised), zeros when there is none
        const int64_t pk = (int64_t)group_prefix_blocks(a, k) * a.block_size;
        n = (int32_t)((pk + a.part_tokens - 1) / a.part_tokens +
                      (max((int64_t)0, T - pk) + a.part_tokens - 1) / a.part_tokens);
    } else if (n <= 1) {
        return;                                  // written directly by the partition kernel
    }
    const int32_t D = a.head_dim;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t cell0 = pair * a.max_parts;
    const float* ml = a.ws_ml + 2 * cell0;
    const float* acc = a.ws_acc + cell0 * D;
    E* out = static_cast<E*>(a.out) + pair * D;

    for (int32_t d0 = 0; d0 < D; d0 += kSlab) {
        const int32_t col = d0 + lane * VEC;
        const bool col_ok = col < D;             // D % VEC == 0: the whole vector is in range
        float m = -INFINITY, l = 0.f, o[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) o[c] = 0.f;
        for (int32_t p0 = warp; p0 < n; p0 += W * kMergeChunk)
            merge_chunk<VEC>(ml, acc, D, col, col_ok, p0, W, n, m, l, o);
        if (lane == 0) {
            m_sm[warp] = m;
            l_sm[warp] = l;
        }
        if constexpr (VEC == 4) {
            *reinterpret_cast<float4*>(&o_sm[warp][lane * 4]) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            o_sm[warp][lane] = o[0];
        }
        __syncthreads();
        // combine the warps' states in warp order, one thread per column
        for (int32_t t = threadIdx.x; t < kSlab && d0 + t < D; t += 32 * W) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, m_sm[w]);
            float L = 0.f, A = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    if (m_sm[w] != -INFINITY) {
                        const float s = exp2f(m_sm[w] - M);
                        L += s * l_sm[w];
                        A += s * o_sm[w][t];
                    }
                }
            }
            out[d0 + t] = Elem<E>::from_float(L > 0.f ? A / L : 0.f);
        }
        __syncthreads();                         // shared state free for the next slab
    }
}

// Warps per merge CTA for a call whose longest sequence has max_parts
// partitions: 2 up to two chunks, 4 up to four, else 8.  (The launch halves
// this while the grid would not fit on the GPU in one wave.)
inline int merge_warps(int32_t max_parts) {
    return max_parts <= 2 * kMergeChunk ? 2 : max_parts <= 4 * kMergeChunk ? 4 : 8;
}

}  // namespace pa
