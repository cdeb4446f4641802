// decode_tiled.cuh -- single-query paged attention on CUDA cores for the
// shapes the TMA + tensor-core kernel does not take: fp32 caches, head dims
// other than 64 and 128 (up to 256, whole 16-byte rows), block sizes that are
// not 8 or a multiple of 16.  Same definition, grid, partitions and workspace
// as the other decode kernels ("vLLM source walkthrough: PagedAttention and
// Continuous Batching" §1.8: per (sequence, head, partition) work, then a
// reduce step across partitions; "Efficient Memory Management for LLM Serving
// with PagedAttention" paper notes, blockwise attention example: one global
// softmax over all blocks).
//
// One CTA of four warps per (partition, kv head x sub-group, sequence); a
// sub-group is up to kTiledHeads query heads of the kv group (more heads take
// more CTAs reading the same K/V, mostly from L2).  The partition's table
// entries are read into shared memory once.  Then every warp runs on its own,
// with no CTA barrier until the end: warp w takes chunks w, w + 4, w + 8, ...
// of CH tokens (16, 8 or 4: about 4 KB of K rows) through its own ring of
// buffers, each with its own mbarrier:
//   - the warp issues a chunk's copies on the bulk-copy engine: a token that
//     starts a run of consecutive valid tokens inside one block copies the
//     run's K rows and V rows (contiguous in the cache) with one cp.async.bulk
//     each; V rows past the length or behind a bad table entry are zeroed;
//   - scores: lane (tq, part) holds tokens tq, tq + 4, ... and the 16-byte
//     pieces part, part + 8, ... of their K rows; the eight lanes of a token
//     read eight neighbouring pieces of one row, so K and q reads are free of
//     bank conflicts, and every q piece read serves CH / 4 tokens.  q sits in
//     shared memory scaled by scale log2(e), so scores come out in base 2;
//   - online softmax of the chunk per head (running max m, sum l, rescale a),
//     the same in every lane;
//   - P V: lane l owns columns [C l, C l + C) (C = 4, or 8 past 128 columns)
//     of every head's accumulator, acc = a acc + sum_t p[h][t] V[t][:].
// At the end the four warps' (m, l, acc) are merged through shared memory,
// into the output or a partition partial for the log-sum-exp merge.
// Every wait is bounded: a timeout raises PA_DEVERR_TIMEOUT, and the warp
// waits (bounded) for its copies in flight before it stops.
#pragma once

#include <algorithm>

#include "decode_generic.cuh"

namespace pa {

constexpr int kTiledWarps = 4;
constexpr int kTiledThreads = 32 * kTiledWarps;
constexpr int kTiledHeads = 8;        // query heads per CTA
// Chunks per warp in shared memory.  Two, so that more CTAs fit on an SM:
// the copy in flight during a chunk's arithmetic keeps HBM busy as long as
// enough warps are resident (a third buffer cost 14-22% of the throughput).
constexpr int kTiledStages = 2;
constexpr int kTiledMaxChunk = 16;
constexpr int kTiledMaxIds = 512;     // table entries of a partition held in shared memory

// Query heads one CTA carries for a group of `group` heads, and that count
// rounded up to 1, 2, 4 or 8 (the kernel's template argument; the extra heads
// have zero q and are not written).
inline int32_t tiled_sub_group(int32_t group) { return group < kTiledHeads ? group : kTiledHeads; }
inline int32_t tiled_heads_rounded(int32_t heads) {
    return heads <= 1 ? 1 : heads <= 2 ? 2 : heads <= 4 ? 4 : 8;
}

// Tokens per chunk: as many of 16, 8 or 4 as 4 KB of K rows hold (bf16:
// 16 up to D = 128, else 8; fp32: 16 up to D = 64, 8 up to 128, else 4).
// Against 2 KB or 3 KB chunks, 4 KB was 3-50% faster on every shape
// measured: the per-chunk wait, table lookup and softmax shuffles are then
// spread over more tokens, while the two-buffer rings still leave room for
// two or more CTAs per SM.
constexpr int kTiledChunkBytes = 4096;
__host__ __device__ inline int32_t tiled_chunk(int32_t head_dim, int32_t elem) {
    const int32_t rows = kTiledChunkBytes / (head_dim * elem);
    return rows >= 16 ? 16 : rows >= 8 ? 8 : 4;
}

// Accumulator columns per lane: 4 up to 128 columns, else 8.
inline int32_t tiled_cols(int32_t head_dim) { return head_dim <= 128 ? 4 : 8; }

// Dynamic shared memory: the warps' rings (reused for the cross-warp merge at
// the end), then q of the (rounded) heads.
inline size_t tiled_smem_bytes(int32_t head_dim, int32_t elem, int32_t heads_rounded) {
    const size_t ring = (size_t)kTiledWarps * kTiledStages * 2 * tiled_chunk(head_dim, elem) *
                        head_dim * elem;
    const size_t merge = (size_t)kTiledWarps * heads_rounded * (head_dim + 2) * 4;
    return std::max(ring, merge) + (size_t)heads_rounded * head_dim * 4;
}

// 1-D bulk copy global -> shared on the copy engine, completion counted on
// `bar`.  Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 16 bytes of shared memory as floats: 8 bf16 or 4 fp32 values.
template <typename E>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int kN = 8;
    __device__ __forceinline__ static void load(const uint8_t* p, float (&v)[8]) {
        const uint4 x = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
    }
};
template <>
struct Vec16<float> {
    static constexpr int kN = 4;
    __device__ __forceinline__ static void load(const uint8_t* p, float (&v)[4]) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
};

// Four consecutive values of a shared-memory row as floats (8- or 16-byte
// aligned).
template <typename E>
__device__ __forceinline__ void load4(const uint8_t* p, float* v) {
    if constexpr (sizeof(E) == 2) {
        const uint2 x = *reinterpret_cast<const uint2*>(p);
        v[0] = __uint_as_float(x.x << 16);
        v[1] = __uint_as_float(x.x & 0xffff0000u);
        v[2] = __uint_as_float(x.y << 16);
        v[3] = __uint_as_float(x.y & 0xffff0000u);
    } else {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
}

// HB: the CTA's heads rounded up to 1, 2, 4 or 8; CH: tokens per chunk;
// C: accumulator columns per lane.
template <typename E, int HB, int CH, int C>
__global__ void __launch_bounds__(kTiledThreads)
decode_tiled_kernel(const DecodeArgs a) {
    static_assert(CH == 4 || CH == 8 || CH == 16, "chunk of 4, 8 or 16 tokens");
    constexpr int TPL = CH / 4;                        // tokens per lane in the scores
    constexpr int kE = (int)sizeof(E);
    constexpr int kV = Vec16<E>::kN;                   // values per 16-byte piece
    constexpr int NQ = kV / 4;                         // float4s of q per piece
    extern __shared__ __align__(128) uint8_t sm_tiled[];
    __shared__ __align__(8) uint64_t sbar[kTiledWarps][kTiledStages];
    __shared__ int32_t fl[kTiledWarps][kTiledStages][kTiledMaxChunk];   // row valid?
    __shared__ __align__(16) float ps[kTiledWarps][HB][CH];               // the chunk's p
    __shared__ int32_t ids[kTiledMaxIds];                                  // partition's table
    __shared__ int32_t s_fail;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t D = a.head_dim;
    constexpr int32_t S = kTiledStages;
    if (tid == 0) {
        for (int32_t w = 0; w < kTiledWarps; ++w)
            for (int32_t s = 0; s < kTiledStages; ++s) mbar_init(smem_u32(&sbar[w][s]), 1);
        mbar_fence_init();
        s_fail = 0;
    }
    griddep_wait();                 // inputs may come from the previous kernel
    const int32_t p = blockIdx.x, i = blockIdx.z;
    const int32_t g = blockIdx.y / a.sub_groups, sg = blockIdx.y - g * a.sub_groups;
    const int32_t Bs = a.block_size, P = a.part_tokens;
    const int32_t H = min(kTiledHeads, a.group - sg * kTiledHeads);   // this CTA's heads
    const int32_t T = checked_len(a, i);
    const int32_t nparts = (int32_t)(((int64_t)T + P - 1) / P);
    const int64_t head0 = (int64_t)i * a.num_q_heads + (int64_t)g * a.group + sg * kTiledHeads;
    E* out = static_cast<E*>(a.out);
    if (T == 0) {          // no visible token: zero output rows
        if (p == 0)
            for (int32_t x = tid; x < H * D; x += kTiledThreads)
                out[head0 * D + x] = Elem<E>::from_float(0.f);
        return;
    }
    if (p >= nparts) return;

    const int32_t t0 = p * P, n = min(P, T - t0);
    const int32_t nchunks = (n + CH - 1) / CH;
    const int32_t rowb = D * kE;                       // bytes of one K or V row
    const int32_t ppr = rowb / 16;                     // 16-byte pieces per row
    const int32_t chunk_bytes = 2 * CH * rowb;
    uint8_t* ring = sm_tiled + warp * S * chunk_bytes;
    const size_t ring_total = (size_t)kTiledWarps * S * chunk_bytes;
    const size_t merge_total = (size_t)kTiledWarps * HB * (D + 2) * 4;
    // q as [head][NQ][piece][4]: the four-value halves of a bf16 piece apart,
    // so eight lanes reading eight neighbouring pieces hit distinct banks
    float* qs = reinterpret_cast<float*>(sm_tiled + (ring_total > merge_total ? ring_total : merge_total));

    const E* q = static_cast<const E*>(a.q);
    const E* kc = static_cast<const E*>(a.k_cache);
    const E* vc = static_cast<const E*>(a.v_cache);
    for (int32_t x = tid; x < HB * D; x += kTiledThreads) {
        const int32_t h = x / D, d = x - h * D;
        const int32_t pc = d / kV, e = d - pc * kV;
        qs[((h * NQ + e / 4) * ppr + pc) * 4 + (e & 3)] =
            h < H ? Elem<E>::to_float(q[head0 * D + x]) * a.scale_log2 : 0.f;
    }
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;
    const int32_t b0 = t0 / Bs, nids = (t0 + n - 1) / Bs - b0 + 1;
    const bool ids_in_smem = nids <= kTiledMaxIds;
    if (ids_in_smem) {
        for (int32_t b = tid; b < nids; b += kTiledThreads) {
            int32_t id = table[b0 + b];
            if (id < 0 || id >= a.num_blocks) {
                raise_error(PA_DEVERR_TABLE_ENTRY);
                id = -1;
            }
            ids[b] = id;
        }
    }
    __syncthreads();

    // ---- every warp on its own: chunks c = warp + 4 j, j < mine ------------
    const int32_t mine = nchunks > warp ? (nchunks - warp + kTiledWarps - 1) / kTiledWarps : 0;

    // Issue the warp's chunk j into buffer j % S.  Lane t < CH looks up token
    // t of the chunk; a lane that starts a run of valid tokens inside one
    // block copies the run's K and V rows; lane 0 arms the buffer's barrier
    // with the bytes; invalid V rows are zeroed (p = 0 must not meet a NaN).
    auto issue = [&](int32_t j) {
        const int32_t c = warp + kTiledWarps * j;
        const int32_t stg = j % S;
        uint8_t* st = ring + stg * chunk_bytes;
        const uint32_t bar = smem_u32(&sbar[warp][stg]);
        const int32_t t = lane, off = c * CH + t, tok = t0 + off;
        int32_t id = -1;
        if (t < CH && off < n) {
            if (ids_in_smem) {
                id = ids[tok / Bs - b0];
            } else {
                id = table[tok / Bs];
                if (id < 0 || id >= a.num_blocks) {
                    raise_error(PA_DEVERR_TABLE_ENTRY);
                    id = -1;
                }
            }
        }
        const bool valid = id >= 0;
        const int32_t blk = tok / Bs;
        const int32_t prev_blk = __shfl_up_sync(0xffffffffu, blk, 1);
        const int32_t prev_valid = __shfl_up_sync(0xffffffffu, (int32_t)valid, 1);
        const bool start = valid && (t == 0 || !prev_valid || prev_blk != blk);
        const uint32_t starts = __ballot_sync(0xffffffffu, start);
        const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
        fence_proxy_async_smem();   // the warp's earlier accesses to the buffer before the copies
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(vmask) * 2u * rowb);
        __syncwarp();
        if (start) {
            // the run ends at the next start or the next invalid token (lanes
            // from CH on are invalid, so t < CH and len <= CH - t)
            const uint32_t stops = (starts | ~vmask) & ~((2u << t) - 1u);
            const int32_t len = __ffs(stops) - 1 - t;
            const int64_t row0 = (((int64_t)id * a.num_kv_heads + g) * Bs + tok % Bs) * D;
            bulk_load(smem_u32(st + t * rowb), kc + row0, (uint32_t)(len * rowb), bar);
            bulk_load(smem_u32(st + (CH + t) * rowb), vc + row0, (uint32_t)(len * rowb), bar);
        }
        uint32_t inv = ~vmask & ((1u << CH) - 1u);
        while (inv) {
            const int32_t r = __ffs(inv) - 1;
            inv &= inv - 1u;
            uint4* vrow = reinterpret_cast<uint4*>(st + (CH + r) * rowb);
            for (int32_t x = lane; x < ppr; x += 32) vrow[x] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (t < CH) fl[warp][stg][t] = valid;
    };

    const int32_t tq = lane >> 3, part = lane & 7;      // scores: token quarter, piece lane
    const int32_t c0 = lane * C;                        // P V: first column of this lane
    const int32_t cnt = max(0, min(C, D - c0));         // 0, 4 or 8 columns (D % 4 == 0)
    float acc[HB][C];
    float m_run[HB], l_run[HB];                         // base-2 running max and sum
#pragma unroll
    for (int32_t h = 0; h < HB; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int32_t x = 0; x < C; ++x) acc[h][x] = 0.f;
    }

    for (int32_t j = 0; j < S && j < mine; ++j) issue(j);
    int32_t issued = min(S, mine);
    for (int32_t j = 0; j < mine; ++j) {
        const int32_t stg = j % S;
        const bool got = mbar_wait_bounded(smem_u32(&sbar[warp][stg]), (j / S) & 1,
                                           kWaitLimitCycles);
        if (__any_sync(0xffffffffu, !got)) {
            // a copy never completed: wait (bounded) for the warp's copies
            // still in flight (one phase per buffer), then stop
            for (int32_t jj = j; jj < issued; ++jj)
                mbar_wait_bounded(smem_u32(&sbar[warp][jj % S]), (jj / S) & 1, kWaitLimitCycles);
            if (lane == 0) s_fail = 1;
            break;
        }
        __syncwarp();               // zeroed rows and flags written by other lanes
        const uint8_t* st = ring + stg * chunk_bytes;

        // scores of tokens tq + 4 u: this lane's pieces, then the sum over the
        // eight piece lanes of each token
        float s[TPL][HB];
#pragma unroll
        for (int32_t u = 0; u < TPL; ++u)
#pragma unroll
            for (int32_t h = 0; h < HB; ++h) s[u][h] = 0.f;
        for (int32_t pc = part; pc < ppr; pc += 8) {
            float k[TPL][kV];
#pragma unroll
            for (int32_t u = 0; u < TPL; ++u)
                Vec16<E>::load(st + (tq + 4 * u) * rowb + pc * 16, k[u]);
#pragma unroll
            for (int32_t h = 0; h < HB; ++h) {
#pragma unroll
                for (int32_t e4 = 0; e4 < NQ; ++e4) {
                    const float4 qv =
                        *reinterpret_cast<const float4*>(qs + ((h * NQ + e4) * ppr + pc) * 4);
#pragma unroll
                    for (int32_t u = 0; u < TPL; ++u) {
                        float x = s[u][h];
                        x = fmaf(qv.x, k[u][4 * e4], x);
                        x = fmaf(qv.y, k[u][4 * e4 + 1], x);
                        x = fmaf(qv.z, k[u][4 * e4 + 2], x);
                        x = fmaf(qv.w, k[u][4 * e4 + 3], x);
                        s[u][h] = x;
                    }
                }
            }
        }
#pragma unroll
        for (int32_t u = 0; u < TPL; ++u) {
            const bool valid = fl[warp][stg][tq + 4 * u] != 0;
#pragma unroll
            for (int32_t h = 0; h < HB; ++h) {
                float x = s[u][h];
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                s[u][h] = valid ? x : -INFINITY;   // a stale K row may hold anything
            }
        }

        // online softmax per head over the chunk (tokens spread over u and
        // the four token quarters); p overwrites s
        float al[HB];
#pragma unroll
        for (int32_t h = 0; h < HB; ++h) {
            float mx = s[0][h];
#pragma unroll
            for (int32_t u = 1; u < TPL; ++u) mx = fmaxf(mx, s[u][h]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[h], mx);
            const float mref = mn == -INFINITY ? 0.f : mn;    // no finite score yet
            al[h] = exp2f(m_run[h] - mref);                   // 0 while m_run = -inf
            float sum = 0.f;
#pragma unroll
            for (int32_t u = 0; u < TPL; ++u) {
                s[u][h] = exp2f(s[u][h] - mref);              // 0 for invalid tokens
                sum += s[u][h];
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            l_run[h] = l_run[h] * al[h] + sum;
            m_run[h] = mn;
        }
        // piece lane h of each token quarter publishes head h's p
#pragma unroll
        for (int32_t h = 0; h < HB; ++h)
            if (part == h)
#pragma unroll
                for (int32_t u = 0; u < TPL; ++u) ps[warp][h][tq + 4 * u] = s[u][h];
        __syncwarp();

        // P V on this lane's columns
#pragma unroll
        for (int32_t h = 0; h < HB; ++h)
#pragma unroll
            for (int32_t x = 0; x < C; ++x) acc[h][x] *= al[h];
        const uint8_t* vcol = st + CH * rowb + c0 * kE;
#pragma unroll 2
        for (int32_t t4 = 0; t4 < CH; t4 += 4) {
            float v[4][C];
#pragma unroll
            for (int32_t u = 0; u < 4; ++u)
#pragma unroll
                for (int32_t x4 = 0; x4 < C; x4 += 4) {
                    if (x4 < cnt) {
                        load4<E>(vcol + (t4 + u) * rowb + x4 * kE, &v[u][x4]);
                    } else {
                        v[u][x4] = v[u][x4 + 1] = v[u][x4 + 2] = v[u][x4 + 3] = 0.f;
                    }
                }
#pragma unroll
            for (int32_t h = 0; h < HB; ++h) {
                const float4 pv = *reinterpret_cast<const float4*>(&ps[warp][h][t4]);
#pragma unroll
                for (int32_t x = 0; x < C; ++x)
                    acc[h][x] = fmaf(pv.w, v[3][x],
                                fmaf(pv.z, v[2][x], fmaf(pv.y, v[1][x], fmaf(pv.x, v[0][x], acc[h][x]))));
            }
        }
        __syncwarp();               // the buffer and p are free
        if (j + S < mine) {
            issue(j + S);
            issued = j + S + 1;
        }
    }

    griddep_launch_dependents();   // the merge kernel may be scheduled now
    __syncthreads();               // every warp is done with its ring
    if (s_fail) {
        if (tid == 0) raise_error(PA_DEVERR_TIMEOUT);
        return;                    // outputs left alone
    }

    // ---- merge the four warps' (m, l, acc) through shared memory ------------
    float* mw = reinterpret_cast<float*>(sm_tiled);     // [warp][HB][D]
    float* mlw = mw + kTiledWarps * HB * D;             // [warp][HB] x (m, l)
#pragma unroll
    for (int32_t h = 0; h < HB; ++h) {
        float* dst = mw + (warp * HB + h) * D + c0;
#pragma unroll
        for (int32_t x4 = 0; x4 < C; x4 += 4)
            if (x4 < cnt)
                *reinterpret_cast<float4*>(dst + x4) =
                    make_float4(acc[h][x4], acc[h][x4 + 1], acc[h][x4 + 2], acc[h][x4 + 3]);
        if (lane == 0) {
            mlw[(warp * HB + h) * 2] = m_run[h];
            mlw[(warp * HB + h) * 2 + 1] = l_run[h];
        }
    }
    __syncthreads();
    for (int32_t x = tid; x < H * D; x += kTiledThreads) {
        const int32_t h = x / D, d = x - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int32_t w = 0; w < kTiledWarps; ++w) M = fmaxf(M, mlw[(w * HB + h) * 2]);
        const float Mr = M == -INFINITY ? 0.f : M;
        float l = 0.f, o = 0.f;
#pragma unroll
        for (int32_t w = 0; w < kTiledWarps; ++w) {
            const float wt = exp2f(mlw[(w * HB + h) * 2] - Mr);   // 0 for a warp with no token
            l = fmaf(mlw[(w * HB + h) * 2 + 1], wt, l);
            o = fmaf(mw[(w * HB + h) * D + d], wt, o);
        }
        if (nparts == 1) {
            out[(head0 + h) * D + d] = Elem<E>::from_float(l > 0.f ? o / l : 0.f);
        } else {
            const int64_t cell = (head0 + h) * a.max_parts + p;
            a.ws_acc[cell * D + d] = o;
            if (d == 0) {
                a.ws_ml[2 * cell] = M;
                a.ws_ml[2 * cell + 1] = l;
            }
        }
    }
}

}  // namespace pa
