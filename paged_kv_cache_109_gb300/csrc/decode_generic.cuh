// decode_generic.cuh -- portable paged decode kernel (fp32 or bf16, any head
// dim, block size and group size).  Used for fp32 caches and for shapes the
// TMA + tensor-core kernel does not cover.
//
// One CTA per (partition p, kv head g, sequence i).  Its three phases follow
// the per-block walk of "vLLM source walkthrough: PagedAttention and
// Continuous Batching" §1.8: (1) for every token of the partition, look up the
// physical block through the table and store the scaled q.k score of each of
// the group's query heads; (2) per head, take the max and turn scores into
// weights 2^(s - m); (3) accumulate the weighted V rows.  A sequence that fits
// one partition writes its output directly; otherwise the partition writes
// (acc, m, l) to the workspace for the log-sum-exp merge (V2 "reduce").
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace pa {

struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    void* out;
    float* ws_acc;
    float* ws_ml;
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t max_seq_len;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t num_blocks;
    int32_t block_size;
    int32_t head_dim;
    int32_t part_tokens;
    int32_t max_parts;
    int32_t sub_groups;   // tensor-core kernel: CTAs per kv head, 16 query heads each
    float scale_log2;     // scale * log2(e)
    // Shared-prefix decode (nullptr / 0 otherwise): group of each sequence
    // (-1: none), the groups' member lists (CSR) and shared leading blocks.
    const int32_t* seq_group;
    const int32_t* member_start;
    const int32_t* members;
    const int32_t* prefix_blocks;
    int32_t num_groups;
    int32_t max_group_size;
    int32_t max_prefix_blocks;
    int32_t prefix_ztiles;   // grid z per group taken by its prefix CTAs
    int32_t prefix_z;        // num_groups * prefix_ztiles: z below this is a prefix CTA
    // Decode with the append fused in (TMA kernel only; nullptr otherwise):
    // sequence i's newest token, at position seq_lens[i] - 1, has K and V rows
    // k_new[i], v_new[i] ([num_seqs, Hkv, head_dim]); the kernel attends to
    // them in place of the cache's old contents of that slot and stores them
    // to the caches.
    const void* k_new;
    const void* v_new;
};

// Shared leading blocks of group k, clamped to the host bound (an entry past
// it is reported and read as 0).
__device__ __forceinline__ int32_t group_prefix_blocks(const DecodeArgs& a, int32_t k) {
    const int32_t b = a.prefix_blocks[k];
    if (b < 0 || b > a.max_prefix_blocks) {
        if (threadIdx.x == 0) raise_error(PA_DEVERR_GROUP);
        return 0;
    }
    return b;
}

// Group of sequence i in a shared-prefix call (-1: none); an id outside
// [0, num_groups) is reported and read as -1.
__device__ __forceinline__ int32_t seq_group_of(const DecodeArgs& a, int32_t i) {
    if (a.seq_group == nullptr) return -1;
    const int32_t k = a.seq_group[i];
    if (k >= a.num_groups) {
        if (threadIdx.x == 0) raise_error(PA_DEVERR_GROUP);
        return -1;
    }
    return k < 0 ? -1 : k;
}

// Effective length from a raw seq_lens value: clamps (and reports) lengths
// the table or the host bound cannot cover.
template <typename Args>
__device__ __forceinline__ int32_t clamp_len(const Args& a, int32_t t) {
    const int64_t cap64 = (int64_t)a.max_blocks * a.block_size;
    const int32_t cap = (int32_t)min((int64_t)a.max_seq_len, cap64);
    if (t < 0 || t > cap) {
        if (threadIdx.x == 0) raise_error(PA_DEVERR_SEQ_LEN);
        t = t < 0 ? 0 : cap;
    }
    return t;
}

// Effective length of sequence i.
__device__ __forceinline__ int32_t checked_len(const DecodeArgs& a, int32_t i) {
    return clamp_len(a, a.seq_lens[i]);
}

template <typename E>
__global__ void __launch_bounds__(128)
decode_generic_kernel(const DecodeArgs a) {
    extern __shared__ float sm_generic[];
    griddep_wait();                 // inputs may come from the previous kernel
    const int32_t p = blockIdx.x, g = blockIdx.y, i = blockIdx.z;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t G = a.group, D = a.head_dim, Bs = a.block_size, P = a.part_tokens;
    const int32_t T = checked_len(a, i);
    const int32_t nparts = (int32_t)(((int64_t)T + P - 1) / P);
    const E* q = static_cast<const E*>(a.q);
    const E* kc = static_cast<const E*>(a.k_cache);
    const E* vc = static_cast<const E*>(a.v_cache);
    E* out = static_cast<E*>(a.out);
    const int64_t head0 = (int64_t)i * a.num_q_heads + (int64_t)g * G;

    if (T == 0) {          // no visible token: zero output row
        if (p == 0)
            for (int32_t x = tid; x < G * D; x += blockDim.x)
                out[head0 * D + x] = Elem<E>::from_float(0.f);
        return;
    }
    if (p >= nparts) return;

    const int32_t t0 = p * P;
    const int32_t n = min(P, T - t0);
    const int32_t nblk = (n + Bs - 1) / Bs;
    // shared: scores/weights [G][P] | q [G][D] | m,l [G][2] | block ids [nblk]
    float* s = sm_generic;
    float* qs = s + (size_t)G * P;
    float* ml = qs + (size_t)G * D;
    int32_t* ids = reinterpret_cast<int32_t*>(ml + 2 * G);

    for (int32_t x = tid; x < G * D; x += blockDim.x)
        qs[x] = Elem<E>::to_float(q[head0 * D + x]);
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks + t0 / Bs;
    for (int32_t b = tid; b < nblk; b += blockDim.x) {
        int32_t id = table[b];
        if (id < 0 || id >= a.num_blocks) {
            raise_error(PA_DEVERR_TABLE_ENTRY);
            id = -1;
        }
        ids[b] = id;
    }
    __syncthreads();

    // (1) scores, one warp per token
    for (int32_t t = warp; t < n; t += blockDim.x / 32) {
        const int32_t id = ids[t / Bs];
        const E* krow = kc + (((int64_t)max(id, 0) * a.num_kv_heads + g) * Bs + t % Bs) * D;
        for (int32_t h = 0; h < G; ++h) {
            float acc = 0.f;
            if (id >= 0)
                for (int32_t d = lane; d < D; d += 32)
                    acc += qs[h * D + d] * Elem<E>::to_float(krow[d]);
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) s[(size_t)h * P + t] = id >= 0 ? acc * a.scale_log2 : -INFINITY;
        }
    }
    __syncthreads();

    // (2) per-head max and weights
    for (int32_t h = warp; h < G; h += blockDim.x / 32) {
        float m = -INFINITY;
        for (int32_t t = lane; t < n; t += 32) m = fmaxf(m, s[(size_t)h * P + t]);
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float l = 0.f;
        for (int32_t t = lane; t < n; t += 32) {
            const float w = m == -INFINITY ? 0.f : exp2f(s[(size_t)h * P + t] - m);
            s[(size_t)h * P + t] = w;
            l += w;
        }
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
            ml[2 * h] = m;
            ml[2 * h + 1] = l;
        }
    }
    __syncthreads();

    // (3) weighted V rows
    griddep_launch_dependents();    // the merge may be scheduled now
    for (int32_t x = tid; x < G * D; x += blockDim.x) {
        const int32_t h = x / D, d = x - h * D;
        float acc = 0.f;
        for (int32_t t = 0; t < n; ++t) {
            const int32_t id = ids[t / Bs];
            if (id < 0) continue;
            const E* vrow = vc + (((int64_t)id * a.num_kv_heads + g) * Bs + t % Bs) * D;
            acc += s[(size_t)h * P + t] * Elem<E>::to_float(vrow[d]);
        }
        const float l = ml[2 * h + 1];
        if (nparts == 1) {
            out[(head0 + h) * D + d] = Elem<E>::from_float(l > 0.f ? acc / l : 0.f);
        } else {
            const int64_t cell = (head0 + h) * a.max_parts + p;
            a.ws_acc[cell * D + d] = acc;
            if (d == 0) {
                a.ws_ml[2 * cell] = ml[2 * h];
                a.ws_ml[2 * cell + 1] = l;
            }
        }
    }
}

// Shared bytes of decode_generic_kernel for a partition of P tokens.
inline size_t generic_smem_bytes(int32_t G, int32_t D, int32_t P, int32_t Bs) {
    return sizeof(float) * ((size_t)G * P + (size_t)G * D + 2 * (size_t)G) +
           sizeof(int32_t) * (size_t)((P + Bs - 1) / Bs);
}

}  // namespace pa
