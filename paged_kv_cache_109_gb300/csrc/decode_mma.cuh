// decode_mma.cuh -- bf16 single-query paged attention on the warp-level
// tensor cores (mma.sync m16n8k16) for the shapes the TMA kernel does not
// take: head dims other than 64 and 128 that are multiples of 16 (up to 128),
// and block sizes other than 8 or a multiple of 16.  Same definition, grid,
// partitions, workspace and merge as the other decode kernels ("vLLM source
// walkthrough: PagedAttention and Continuous Batching" §1.8: per (sequence,
// head, partition) work through the block table, then a reduce step across
// partitions; "Efficient Memory Management for LLM Serving with
// PagedAttention" paper notes, blockwise attention example).
//
// One CTA of four warps per (partition, kv head x sub-group of 16 query
// heads, sequence).  Warp w takes the partition's 16-token chunks w, w + 4,
// ... through its own two-stage ring.  Each token's K row and V row is one
// bulk copy (lane r copies row r's K, lane 16 + r its V), so blocks of any
// size work and every row can be padded by 16 bytes: the eight rows an
// ldmatrix reads then fall in eight bank groups.  A stage's copies are
// counted on its own mbarrier; the warp waits on its own stages, with no CTA
// barrier until the end, and every wait is bounded.  Per chunk, with the sub-group's query heads as the
// 16 rows of the MMA tile (rows past G zero):
//   S[16 x 16] = Q . K^T, online softmax in base 2, acc += P . V
// with P split into bf16 hi + lo parts as in the TMA kernel (G <= 8: the lo
// parts ride in rows 8-15; G > 8: a second product).  The four warps'
// (m, l, acc) are merged through shared memory at the end.
#pragma once

#include "decode_tiled.cuh"

namespace pa {

constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kMmaChunk = 16;     // tokens per chunk
// Chunks per warp in shared memory.  Two, with launch bounds of three CTAs
// per SM: the kernel is latency-bound, and three stages held it to two CTAs
// per SM (0.43-0.45 against 0.52-0.55 of the copy peak at G = 16, D = 112 and
// G = 5, D = 96).
constexpr int kMmaStages = 2;
constexpr int kMmaMaxDim = 128;

// Dynamic shared memory: the warps' rings, reused at the end for the
// cross-warp merge (m, l and acc of 16 rows per warp).
inline size_t decode_mma_smem_bytes(int32_t head_dim) {
    const size_t stride = (size_t)head_dim * 2 + 16;
    const size_t ring = (size_t)kMmaWarps * kMmaStages * 2 * kMmaChunk * stride;
    const size_t merge = (size_t)kMmaWarps * 16 * (head_dim + 2) * 4;
    return std::max(ring, merge);
}

template <bool G16>
__global__ void __launch_bounds__(kMmaThreads, 3)
decode_mma_kernel(const DecodeArgs a) {
    constexpr int KS = kMmaMaxDim / 16;   // k steps of S (at most)
    constexpr int DT = kMmaMaxDim / 8;    // n-tiles of acc (at most)
    extern __shared__ __align__(128) uint8_t sm_dm[];
    __shared__ __align__(8) uint64_t sbar[kMmaWarps][kMmaStages];
    __shared__ int32_t fl[kMmaWarps][kMmaStages][kMmaChunk];   // token valid?
    __shared__ int32_t ids[kTiledMaxIds];                        // the partition's table entries
    __shared__ int32_t s_fail;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int32_t w = 0; w < kMmaWarps; ++w)
            for (int32_t s2 = 0; s2 < kMmaStages; ++s2) mbar_init(smem_u32(&sbar[w][s2]), 1);
        mbar_fence_init();
        s_fail = 0;
    }
    griddep_wait();                          // inputs may come from the previous kernel
    const int32_t grp = lane >> 2, tig = lane & 3;
    const int32_t lm = lane >> 3, lr = lane & 7;   // ldmatrix: matrix, row in matrix
    const int32_t D = a.head_dim, Bs = a.block_size, P = a.part_tokens;
    const int32_t p = blockIdx.x, i = blockIdx.z;
    const int32_t g = blockIdx.y / a.sub_groups, sg = blockIdx.y - g * a.sub_groups;
    const int32_t G = min(16, a.group - sg * 16);           // this CTA's query heads
    const int32_t T = checked_len(a, i);
    const int32_t nparts = (int32_t)(((int64_t)T + P - 1) / P);
    const int64_t head0 = (int64_t)i * a.num_q_heads + (int64_t)g * a.group + sg * 16;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    if (T == 0) {          // no visible token: zero output rows
        if (p == 0)
            for (int32_t x = tid; x < G * D; x += kMmaThreads)
                out[head0 * D + x] = __float2bfloat16_rn(0.f);
        return;
    }
    if (p >= nparts) return;

    const int32_t t0 = p * P, n = min(P, T - t0);
    const int32_t nchunks = (n + kMmaChunk - 1) / kMmaChunk;
    const int32_t rowb = D * 2, stride = rowb + 16, ppr = rowb / 16;
    const int32_t stage_bytes = 2 * kMmaChunk * stride;     // K rows, then V rows
    const uint32_t ring = smem_u32(sm_dm) + warp * kMmaStages * stage_bytes;

    // the partition's table entries, checked once (longer partitions read
    // the table as they go)
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;
    const int32_t b0 = t0 / Bs, nids = (t0 + n - 1) / Bs - b0 + 1;
    const bool ids_in_smem = nids <= kTiledMaxIds;
    if (ids_in_smem) {
        for (int32_t b = tid; b < nids; b += kMmaThreads) {
            int32_t id = table[b0 + b];
            if (id < 0 || id >= a.num_blocks) {
                raise_error(PA_DEVERR_TABLE_ENTRY);
                id = -1;
            }
            ids[b] = id;
        }
    }

    // Q fragments (A operand): rows = the sub-group's query heads, k = head dim
    uint32_t qa[KS][4];
    {
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
        const bool r0 = grp < G, r1 = G16 && grp + 8 < G;
        const __nv_bfloat16* q0 = q + (head0 + grp) * D;
        const __nv_bfloat16* q1 = q + (head0 + grp + 8) * D;
#pragma unroll
        for (int32_t ks = 0; ks < KS; ++ks) {
            const int32_t d0 = ks * 16 + 2 * tig;
            const bool in = ks < D / 16;
            qa[ks][0] = in && r0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
            qa[ks][1] = in && r1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
            qa[ks][2] = in && r0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
            qa[ks][3] = in && r1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
        }
    }
    __syncthreads();       // ids

    // Issue the warp's chunk j into stage j % kMmaStages.  Lane r < 16 looks
    // up token r of the chunk and copies its K row, lane 16 + r its V row;
    // lane 0 arms the stage's barrier with the bytes.  V rows of tokens past
    // the partition or behind a bad table entry are zeroed (p = 0 must not
    // meet a NaN), and their scores are masked by the stage's flags.
    const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
    const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
    const int32_t mine = nchunks > warp ? (nchunks - warp + kMmaWarps - 1) / kMmaWarps : 0;
    auto issue = [&](int32_t j) {
        const int32_t c = warp + kMmaWarps * j;
        const int32_t stg = j % kMmaStages;
        const uint32_t kb = ring + stg * stage_bytes;
        const uint32_t bar = smem_u32(&sbar[warp][stg]);
        const int32_t r = lane & 15;
        const int32_t off = c * kMmaChunk + r, tok = t0 + off;
        int32_t id = -1;
        if (off < n) {
            if (ids_in_smem) {
                id = ids[tok / Bs - b0];
            } else {
                id = table[tok / Bs];
                if (id < 0 || id >= a.num_blocks) {
                    if (lane < 16) raise_error(PA_DEVERR_TABLE_ENTRY);
                    id = -1;
                }
            }
        }
        const bool valid = id >= 0;
        const uint32_t vmask = __ballot_sync(0xffffffffu, valid) & 0xffffu;
        fence_proxy_async_smem();   // the warp's earlier accesses to the stage before the copies
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(vmask) * 2u * rowb);
        __syncwarp();
        if (valid) {
            const int64_t row = (((int64_t)id * a.num_kv_heads + g) * Bs + tok % Bs) * D;
            const __nv_bfloat16* src = lane < 16 ? kc + row : vc + row;
            bulk_load(kb + (lane < 16 ? 0 : kMmaChunk * stride) + r * stride, src, (uint32_t)rowb,
                      bar);
        }
        uint32_t inv = ~vmask & 0xffffu;
        uint8_t* vgen = sm_dm + warp * kMmaStages * stage_bytes + stg * stage_bytes +
                        kMmaChunk * stride;
        while (inv) {
            const int32_t rr = __ffs(inv) - 1;
            inv &= inv - 1u;
            uint4* vrow = reinterpret_cast<uint4*>(vgen + rr * stride);
            for (int32_t x = lane; x < ppr; x += 32) vrow[x] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (lane < 16) fl[warp][stg][r] = valid;
    };

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[DT][4];
#pragma unroll
    for (int32_t nd = 0; nd < DT; ++nd) acc[nd][0] = acc[nd][1] = acc[nd][2] = acc[nd][3] = 0.f;

    for (int32_t j = 0; j < kMmaStages && j < mine; ++j) issue(j);
    int32_t issued = min(kMmaStages, mine);
    for (int32_t j = 0; j < mine; ++j) {
        const int32_t stg = j % kMmaStages;
        const bool got = mbar_wait_bounded(smem_u32(&sbar[warp][stg]), (j / kMmaStages) & 1,
                                           kWaitLimitCycles);
        if (__any_sync(0xffffffffu, !got)) {
            // a copy never completed: wait (bounded) for the warp's copies
            // still in flight (one phase per stage), then stop
            for (int32_t jj = j; jj < issued; ++jj)
                mbar_wait_bounded(smem_u32(&sbar[warp][jj % kMmaStages]), (jj / kMmaStages) & 1,
                                  kWaitLimitCycles);
            if (lane == 0) s_fail = 1;
            break;
        }
        __syncwarp();              // zeroed rows and flags written by other lanes
        const int32_t c = warp + kMmaWarps * j;
        const uint32_t kb = ring + stg * stage_bytes;
        const uint32_t vb = kb + kMmaChunk * stride;
        const int32_t nvalid = min(kMmaChunk, n - c * kMmaChunk);

        // S = Q . K^T for the 16 tokens of the chunk (two n-tiles of 8)
        float s[2][4];
#pragma unroll
        for (int32_t nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int32_t ks = 0; ks < KS; ++ks) {
            if (ks < D / 16) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kb + ((lm >> 1) * 8 + lr) * stride + (ks * 16 + (lm & 1) * 8) * 2,
                        b0, b1, b2, b3);
                mma_bf16_16816(s[0], qa[ks], b0, b1);
                mma_bf16_16816(s[1], qa[ks], b2, b3);
            }
        }
        // scale, mask, online softmax of rows grp (and grp + 8 with G16)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int32_t nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int32_t e = 0; e < 2; ++e) {
                const int32_t col = nt * 8 + 2 * tig + e;
                const bool valid = col < nvalid && fl[warp][stg][col] != 0;
                s[nt][e] = valid ? s[nt][e] * a.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][e]);
                if (G16) {
                    s[nt][2 + e] = valid ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        // a chunk whose tokens all sit behind bad table entries has no finite
        // score: the reference is then 0, which leaves everything at 0
        const float mn0 = fmaxf(m0, mx0);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
        const float al0 = exp2f(m0 - ref0);
        m0 = mn0;
        float al1 = 1.f, ref1 = 0.f;
        if (G16) {
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn1 = fmaxf(m1, mx1);
            ref1 = mn1 == -INFINITY ? 0.f : mn1;
            al1 = exp2f(m1 - ref1);
            m1 = mn1;
        }
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int32_t nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int32_t e = 0; e < 2; ++e) {
                s[nt][e] = exp2f(s[nt][e] - ref0);
                rs0 += s[nt][e];
                if (G16) {
                    s[nt][2 + e] = exp2f(s[nt][2 + e] - ref1);
                    rs1 += s[nt][2 + e];
                }
            }
        l0 = l0 * al0 + rs0;
        if (G16) l1 = l1 * al1 + rs1;
#pragma unroll
        for (int32_t nd = 0; nd < DT; ++nd) {
            acc[nd][0] *= al0;
            acc[nd][1] *= al0;
            acc[nd][2] *= G16 ? al1 : al0;      // G <= 8: the lo products of rows 0-7
            acc[nd][3] *= G16 ? al1 : al0;
        }

        // acc += P . V with P = hi + lo (both bf16)
        uint32_t pf[4], pl[4];
        auto split = [](float x, float y, uint32_t& hi, uint32_t& lo) {
            hi = pack_bf16x2(x, y);
            lo = pack_bf16x2(x - __uint_as_float(hi << 16), y - __uint_as_float(hi & 0xffff0000u));
        };
        split(s[0][0], s[0][1], pf[0], pl[0]);
        split(s[1][0], s[1][1], pf[2], pl[2]);
        if (G16) {
            split(s[0][2], s[0][3], pf[1], pl[1]);
            split(s[1][2], s[1][3], pf[3], pl[3]);
        } else {
            pf[1] = pl[0];
            pf[3] = pl[2];
        }
#pragma unroll
        for (int32_t dp = 0; dp < KS; ++dp) {
            if (dp < D / 16) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vb + ((lm & 1) * 8 + lr) * stride + (dp * 16 + (lm >> 1) * 8) * 2,
                              b0, b1, b2, b3);
                mma_bf16_16816(acc[2 * dp], pf, b0, b1);
                mma_bf16_16816(acc[2 * dp + 1], pf, b2, b3);
                if (G16) {
                    mma_bf16_16816(acc[2 * dp], pl, b0, b1);
                    mma_bf16_16816(acc[2 * dp + 1], pl, b2, b3);
                }
            }
        }
        __syncwarp();              // the stage is free for chunk j + kMmaStages
        if (j + kMmaStages < mine) {
            issue(j + kMmaStages);
            issued = j + kMmaStages + 1;
        }
    }
    griddep_launch_dependents();   // the merge kernel may be scheduled now

    if (!G16) {            // the lo products of rows 0-7 landed in rows 8-15
#pragma unroll
        for (int32_t nd = 0; nd < DT; ++nd) {
            acc[nd][0] += acc[nd][2];
            acc[nd][1] += acc[nd][3];
        }
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    if (G16) {
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    __syncthreads();       // every warp is done with its ring
    if (s_fail) {
        if (tid == 0) raise_error(PA_DEVERR_TIMEOUT);
        return;            // outputs left alone
    }

    // merge the four warps' (m, l, acc) through shared memory
    float* cm = reinterpret_cast<float*>(sm_dm);     // [warp][16]
    float* cl = cm + kMmaWarps * 16;                 // [warp][16]
    float* ca = cl + kMmaWarps * 16;                 // [warp][16][D]
    if (tig == 0) {
        cm[warp * 16 + grp] = m0;
        cl[warp * 16 + grp] = l0;
        if (G16) {
            cm[warp * 16 + grp + 8] = m1;
            cl[warp * 16 + grp + 8] = l1;
        }
    }
#pragma unroll
    for (int32_t nd = 0; nd < DT; ++nd) {
        if (nd < D / 8) {
            const int32_t d = nd * 8 + 2 * tig;
            float* r0 = ca + (warp * 16 + grp) * D + d;
            r0[0] = acc[nd][0];
            r0[1] = acc[nd][1];
            if (G16) {
                float* r1 = ca + (warp * 16 + grp + 8) * D + d;
                r1[0] = acc[nd][2];
                r1[1] = acc[nd][3];
            }
        }
    }
    __syncthreads();
    for (int32_t x = tid; x < G * D; x += kMmaThreads) {
        const int32_t h = x / D, d = x - h * D;
        float M = -INFINITY, L = 0.f, A = 0.f;
#pragma unroll
        for (int32_t w = 0; w < kMmaWarps; ++w) M = fmaxf(M, cm[w * 16 + h]);
#pragma unroll
        for (int32_t w = 0; w < kMmaWarps; ++w) {
            const float mw = cm[w * 16 + h];
            if (mw != -INFINITY) {         // a warp with no chunk adds nothing
                const float e = exp2f(mw - M);
                L += e * cl[w * 16 + h];
                A += e * ca[(w * 16 + h) * D + d];
            }
        }
        if (nparts == 1) {
            out[(head0 + h) * D + d] = __float2bfloat16_rn(L > 0.f ? A / L : 0.f);
        } else {
            const int64_t cell = (head0 + h) * a.max_parts + p;
            a.ws_acc[cell * D + d] = A;
            if (d == 0) {
                a.ws_ml[2 * cell] = M;
                a.ws_ml[2 * cell + 1] = L;
            }
        }
    }
}

}  // namespace pa
