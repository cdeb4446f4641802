// prefill_tma_mma.cuh -- multi-query (chunked prefill) paged attention, bf16.
//
// Sequence i owns the packed query rows [query_start[i], query_start[i+1]):
// its last L_i positions, row r at position p = T_i - L_i + (r - start),
// attending to keys 0..p ("vLLM source walkthrough: PagedAttention and
// Continuous Batching" §2.8: chunked prefill and decode rows in one batch;
// "vLLM PagedAttention: from memory fragmentation to slot mapping" §6: query
// start locations slice the tokens per request, positions set the causal
// boundary).
//
// One CTA per (query tile, kv head g, sequence i), four warps.  A tile is 64
// MMA rows = (query token, query head of the group) pairs with the head
// fastest, so a tile holds 64/G tokens and every K/V chunk loaded for the
// tile serves all of them.  Thread 0 issues TMA copies of 16-key chunks of
// the sequence's (block, kv head) tiles through the block table into a
// kStages ring; all four warps consume each chunk (S = Q K^T, causal mask,
// online softmax, acc += P V, all on mma.sync bf16 -> fp32) and meet at a
// barrier before the stage is refilled.  Tiles are scheduled latest-first:
// under the causal mask later tiles see more keys.  The table slice lives in
// a sliding shared-memory window, so any context length works.
#pragma once

#include <cuda.h>

#include "decode_generic.cuh"
#include "ptx.cuh"

namespace pa {

#ifndef PA_PREFILL_STAGES
#define PA_PREFILL_STAGES 4
#endif

struct PrefillArgs {
    const void* q;                  // [total_q][Hq][D]
    const void* k_cache;            // [num_blocks][Hkv][B][D] (portable kernel)
    const void* v_cache;
    const int32_t* query_start;     // [N + 1]
    const int32_t* seq_lens;        // [N]
    const int32_t* block_tables;    // [N][max_blocks]
    void* out;                      // [total_q][Hq][D]
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t max_seq_len;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t num_blocks;
    int32_t block_size;
    int32_t head_dim;
    int32_t tokens_per_tile;        // 64 / group
    float scale_log2;
};

template <int D>
struct PrefillCfg {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kRows = 64;                      // MMA rows per CTA
    static constexpr int kChunk = 16;                     // keys per stage
    static constexpr int kBoxCols = 64;
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kBoxBytes = kChunk * 128;
    static constexpr int kTileBytes = kBoxes * kBoxBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = PA_PREFILL_STAGES;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kKSteps = D / 16;
    static constexpr int kDTiles = D / 8;
    static constexpr int kWindow = 1024;                  // block ids kept in shared memory
    static size_t smem_bytes() { return 1024 + kRingBytes + 8 * kStages + 4 * kWindow + 16; }
};

template <int D>
__global__ void __launch_bounds__(128, 3)
prefill_tma_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t sm_raw[];
    __shared__ int s_fail;
    __shared__ int s_stage_ok[C::kStages];
    __shared__ int s_win0;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kRingBytes);
    int32_t* win = reinterpret_cast<int32_t*>(bars + C::kStages);

    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t grp = lane >> 2, tig = lane & 3;
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
        mbar_fence_init();
        s_fail = 0;
    }
    if (tid == 32) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    griddep_wait();

    const int32_t tile = gridDim.x - 1 - blockIdx.x;      // latest (longest) tiles first
    const int32_t g = blockIdx.y, i = blockIdx.z;
    const int32_t G = a.group, BS = a.block_size;
    const int32_t q0 = a.query_start[i], q1 = a.query_start[i + 1];
    const int32_t L = q1 - q0;
    const int32_t T = clamp_len(a, a.seq_lens[i]);
    if (L > T) {
        if (tid == 0 && tile == 0 && g == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int32_t tok0 = tile * a.tokens_per_tile;
    if (L <= 0 || tok0 >= L) return;
    const int32_t ntok = min(a.tokens_per_tile, L - tok0);
    const int32_t pos0 = T - L + tok0;                    // position of the tile's first token
    const int32_t nkeys = pos0 + ntok;                    // keys 0 .. last token's position
    const int32_t nchunk = (nkeys + C::kChunk - 1) / C::kChunk;
    const int32_t nblk = (nkeys + BS - 1) / BS;
    const int32_t cpb = BS >= C::kChunk ? BS / C::kChunk : 1;
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;

    // this thread's two MMA rows (r and r + 8 of its warp's 16)
    const int32_t rA = warp * 16 + grp, rB = rA + 8;
    const int32_t tA = rA / G, hA = rA - tA * G, tB = rB / G, hB = rB - tB * G;
    const bool okA = tA < ntok, okB = tB < ntok;
    // rows past the last token keep Q = 0 and the tile's last position, so
    // their scores stay finite; they are never written
    const int32_t pA = pos0 + (okA ? tA : ntok - 1), pB = pos0 + (okB ? tB : ntok - 1);
    uint32_t qa[C::kKSteps][4];
    {
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
        const __nv_bfloat16* qA = q + ((int64_t)(q0 + tok0 + tA) * a.num_q_heads + g * G + hA) * D;
        const __nv_bfloat16* qB = q + ((int64_t)(q0 + tok0 + tB) * a.num_q_heads + g * G + hB) * D;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            const int d0 = ks * 16 + 2 * tig;
            qa[ks][0] = okA ? *reinterpret_cast<const uint32_t*>(qA + d0) : 0u;
            qa[ks][1] = okB ? *reinterpret_cast<const uint32_t*>(qB + d0) : 0u;
            qa[ks][2] = okA ? *reinterpret_cast<const uint32_t*>(qA + d0 + 8) : 0u;
            qa[ks][3] = okB ? *reinterpret_cast<const uint32_t*>(qB + d0 + 8) : 0u;
        }
    }

    // block-id window [s_win0, s_win0 + kWindow), filled by the whole CTA
    auto fill_window = [&](int32_t first) {
        for (int32_t b = tid; b < C::kWindow; b += C::kThreads) {
            int32_t id = -1;
            if (first + b < nblk) {
                id = table[first + b];
                if (id < 0 || id >= a.num_blocks) {
                    raise_error(PA_DEVERR_TABLE_ENTRY);
                    id = -1;
                }
            }
            win[b] = id;
        }
        if (tid == 0) s_win0 = first;
    };
    auto first_block_of = [&](int32_t c) { return BS >= C::kChunk ? c / cpb : 2 * c; };
    auto last_block_of = [&](int32_t c) {
        return BS >= C::kChunk ? c / cpb : min(2 * c + 1, nblk - 1);
    };

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int32_t c) {   // thread 0 only; the chunk's blocks are in the window
        const int32_t st = c % C::kStages;
        const uint32_t bar = smem_u32(&bars[st]);
        const int32_t w0 = s_win0;
        const int32_t b0 = first_block_of(c), b1 = last_block_of(c);
        bool ok = true;
        for (int32_t b = b0; b <= b1; ++b) ok = ok && win[b - w0] >= 0;
        s_stage_ok[st] = ok;
        if (!ok) {
            mbar_arrive(bar);
            return;
        }
        const uint32_t dst = smem_u32(sm) + st * C::kStageBytes;
        fence_proxy_async_smem();
        if (BS >= C::kChunk) {
            const int32_t y = (c - b0 * cpb) * C::kChunk;
            const int32_t z = win[b0 - w0] * a.num_kv_heads + g;
            mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b)
                tma_load_3d_hint(dst + b * C::kBoxBytes, &tmap_k, b * C::kBoxCols, y, z, bar,
                                 policy);
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b)
                tma_load_3d_hint(dst + C::kTileBytes + b * C::kBoxBytes, &tmap_v,
                                 b * C::kBoxCols, y, z, bar, policy);
        } else {
            const int32_t halves = b1 - b0 + 1;
            mbar_arrive_expect_tx(bar, halves * (C::kStageBytes / 2));
            for (int h = 0; h < halves; ++h) {
                const int32_t z = win[b0 + h - w0] * a.num_kv_heads + g;
#pragma unroll
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d_hint(dst + b * C::kBoxBytes + h * 1024, &tmap_k,
                                     b * C::kBoxCols, 0, z, bar, policy);
#pragma unroll
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d_hint(dst + C::kTileBytes + b * C::kBoxBytes + h * 1024,
                                     &tmap_v, b * C::kBoxCols, 0, z, bar, policy);
            }
        }
    };

    fill_window(0);
    __syncthreads();
    if (tid == 0) {
        const int32_t pre = min(nchunk, C::kStages);
        for (int32_t c = 0; c < pre; ++c) issue(c);
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[C::kDTiles][4];
#pragma unroll
    for (int nd = 0; nd < C::kDTiles; ++nd) acc[nd][0] = acc[nd][1] = acc[nd][2] = acc[nd][3] = 0.f;
    const int32_t lm = lane >> 3, lr = lane & 7;
    bool failed = false;
    int32_t c = 0;

    for (; c < nchunk; ++c) {
        const int32_t st = c % C::kStages;
        const bool ok =
            mbar_wait_bounded(smem_u32(&bars[st]), (c / C::kStages) & 1, kWaitLimitCycles);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (s_stage_ok[st]) {
            const uint32_t kb = smem_u32(sm) + st * C::kStageBytes;
            const uint32_t vb = kb + C::kTileBytes;
            const int32_t key0 = c * C::kChunk;
            const int32_t nvalid = min(C::kChunk, nkeys - key0);
            if (nvalid < C::kChunk) {
                // keys past the last token's position: clear their V rows
                // (their weights are 0, the rows may hold anything)
                if (warp == 0) {
                    uint8_t* vt = sm + st * C::kStageBytes + C::kTileBytes;
                    const int32_t pieces = (C::kChunk - nvalid) * 8;
                    for (int32_t x = lane; x < C::kBoxes * pieces; x += 32) {
                        const int32_t b = x / pieces, r = x - b * pieces;
                        *reinterpret_cast<uint4*>(vt + b * C::kBoxBytes + nvalid * 128 + r * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                __syncthreads();
            }
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            {
                const int tok = (lm >> 1) * 8 + lr;
#pragma unroll
                for (int ks = 0; ks < C::kKSteps; ++ks) {
                    const int ch = ((ks & 3) << 1) + (lm & 1);
                    const uint32_t addr =
                        kb + (ks >> 2) * C::kBoxBytes + tok * 128 + ((ch ^ (tok & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    mma_bf16_16816(s[0], qa[ks], b0, b1);
                    mma_bf16_16816(s[1], qa[ks], b2, b3);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int32_t key = key0 + nt * 8 + 2 * tig + e;
                    s[nt][e] = key <= pA ? s[nt][e] * a.scale_log2 : -INFINITY;
                    s[nt][2 + e] = key <= pB ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
                    mx0 = fmaxf(mx0, s[nt][e]);
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            // a row whose keys are all masked so far keeps m = -inf: no weight
            const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
            const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] = mn0 == -INFINITY ? 0.f : exp2f(s[nt][e] - mn0);
                    s[nt][2 + e] = mn1 == -INFINITY ? 0.f : exp2f(s[nt][2 + e] - mn1);
                    rs0 += s[nt][e];
                    rs1 += s[nt][2 + e];
                }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
#pragma unroll
            for (int nd = 0; nd < C::kDTiles; ++nd) {
                acc[nd][0] *= al0;
                acc[nd][1] *= al0;
                acc[nd][2] *= al1;
                acc[nd][3] *= al1;
            }
            uint32_t pf[4];
            pf[0] = pack_bf16x2(s[0][0], s[0][1]);
            pf[1] = pack_bf16x2(s[0][2], s[0][3]);
            pf[2] = pack_bf16x2(s[1][0], s[1][1]);
            pf[3] = pack_bf16x2(s[1][2], s[1][3]);
            {
                const int tok = (lm & 1) * 8 + lr;
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const int chunk = 2 * dp + (lm >> 1);
                    const uint32_t addr = vb + (chunk >> 3) * C::kBoxBytes + tok * 128 +
                                          (((chunk & 7) ^ (tok & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(addr, b0, b1, b2, b3);
                    mma_bf16_16816(acc[2 * dp], pf, b0, b1);
                    mma_bf16_16816(acc[2 * dp + 1], pf, b2, b3);
                }
            }
        }
        // every warp is done with stage st: refill it with chunk c + kStages
        const int32_t next = c + C::kStages;
        const bool refill = next < nchunk && last_block_of(next) >= s_win0 + C::kWindow;
        __syncthreads();
        if (refill) {                        // uniform: slide the window to the next chunk
            fill_window(first_block_of(next));
            __syncthreads();
        }
        if (tid == 0 && next < nchunk) issue(next);
    }

    if (failed && tid == 0) {
        // let the copies still in flight land (bounded) before the CTA exits
        for (int32_t k = c; k < min(nchunk, c + C::kStages); ++k)
            mbar_wait_bounded(smem_u32(&bars[k % C::kStages]), (k / C::kStages) & 1,
                              kWaitLimitCycles);
        raise_error(PA_DEVERR_TIMEOUT);
        s_fail = 1;
    }
    griddep_launch_dependents();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const float iA = (!failed && l0 > 0.f) ? 1.f / l0 : 0.f;
    const float iB = (!failed && l1 > 0.f) ? 1.f / l1 : 0.f;
    __nv_bfloat16* oA = out + ((int64_t)(q0 + tok0 + tA) * a.num_q_heads + g * G + hA) * D;
    __nv_bfloat16* oB = out + ((int64_t)(q0 + tok0 + tB) * a.num_q_heads + g * G + hB) * D;
#pragma unroll
    for (int nd = 0; nd < C::kDTiles; ++nd) {
        const int d = nd * 8 + 2 * tig;
        if (okA) {
            oA[d] = __float2bfloat16_rn(acc[nd][0] * iA);
            oA[d + 1] = __float2bfloat16_rn(acc[nd][1] * iA);
        }
        if (okB) {
            oB[d] = __float2bfloat16_rn(acc[nd][2] * iB);
            oB[d + 1] = __float2bfloat16_rn(acc[nd][3] * iB);
        }
    }
}

}  // namespace pa
