// prefill_tc.cuh -- multi-query (chunked prefill) paged attention on the
// 5th-generation tensor cores (tcgen05, tensor-memory accumulators), bf16.
//
// Same definition as prefill_tma_mma.cuh: sequence i's packed query rows are
// its last L_i positions, row r at position p attends to keys 0..p
// ("vLLM source walkthrough: PagedAttention and Continuous Batching" §2.8;
// "vLLM PagedAttention: from memory fragmentation to slot mapping" §6).
//
// One CTA per (query tile, kv head g, sequence i); 128 threads; a tile is 128
// MMA rows = (query token, query head of the group) pairs, head fastest, so it
// holds 128/G tokens.  Thread t owns row t: tensor-memory lane t.
//
// Per block of 32 keys (two 16-key chunks fetched by TMA through the block
// table into a 3-stage ring):
//   S = Q K^T       tcgen05.mma M128 N32 (K-major A = Q, K-major B = K chunk,
//                   both 128-byte swizzled), fp32 in tensor memory;
//   softmax         each thread loads its row of S (tcgen05.ld), masks keys
//                   past its position, updates m and l in base 2, writes its
//                   row of P (bf16) to shared memory and, when its row maximum
//                   rose, rescales its row of O in tensor memory;
//   O += P V        tcgen05.mma M128 N64 per 64 output columns (K-major A = P,
//                   MN-major B = V chunk rows).
// Thread 0 issues the copies and the MMAs; commits signal mbarriers.  At the
// end each thread reads its O row, divides by l and stores it.  Two CTAs per
// SM let one CTA's softmax overlap the other's tensor-core work.
#pragma once

#include "prefill_tma_mma.cuh"

namespace pa {

template <int D>
struct PrefillTcCfg {
    static constexpr int kThreads = 128;
    static constexpr int kRows = 128;                    // MMA M = TMEM lanes
    static constexpr int kKeys = 32;                     // keys per block (MMA N of S)
    static constexpr int kChunk = 16;                    // keys per TMA chunk
    static constexpr int kHalves = D / 64;               // 64-column (128-byte) slices
    static constexpr int kBox = kChunk * 128;            // one chunk, one slice: 2 KiB
    static constexpr int kSlice = kKeys * 128;           // one block, one slice: 4 KiB
    static constexpr int kTile = kHalves * kSlice;       // K (or V) block
    static constexpr int kStageBytes = 2 * kTile;        // K + V
    static constexpr int kStages = 4;
    static constexpr int kQSlice = kRows * 128;          // 16 KiB
    static constexpr int kQBytes = kHalves * kQSlice;
    static constexpr int kPBytes = kRows * kKeys * 2;    // 8 KiB, no-swizzle core matrices
    static constexpr int kWindow = 256;                  // block ids in shared memory
    static constexpr uint32_t kTmemCols = 256;           // S: 2 x 32 columns, O: D columns
    static constexpr uint32_t kOCol = 64;
    static constexpr int kQOff = 0;
    static constexpr int kStageOff = kQBytes;
    static constexpr int kPOff = kStageOff + kStages * kStageBytes;
    static constexpr int kBarOff = kPOff + kPBytes;
    static constexpr int kBars = kStages + 4;            // full[kStages], S[2], O, final drain
    static constexpr int kSlotOff = kBarOff + 8 * kBars;
    static constexpr int kWinOff = kSlotOff + 16;
    static size_t smem_bytes() { return 1024 + kWinOff + 4 * kWindow; }
    static_assert(D == 64 || D == 128, "head_dim");
};

template <int D>
__global__ void __launch_bounds__(128, 2)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    using C = PrefillTcCfg<D>;
    extern __shared__ uint8_t sm_raw[];
    __shared__ int s_stage_ok[C::kStages];
    __shared__ int s_win0;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sm_u = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::kSlotOff);
    int32_t* win = reinterpret_cast<int32_t*>(sm + C::kWinOff);
    const uint32_t bar_s0 = smem_u32(&bars[C::kStages]);      // S buffer 0, buffer 1 at +8
    const uint32_t bar_o = smem_u32(&bars[C::kStages + 2]);
    const uint32_t bar_fin = smem_u32(&bars[C::kStages + 3]);

    const int32_t tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < C::kBars; ++s) mbar_init(smem_u32(&bars[s]), 1);
        mbar_fence_init();
    }
    if (tid == 32) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    griddep_wait();

    const int32_t tile = gridDim.x - 1 - blockIdx.x;      // latest (longest) tiles first
    const int32_t g = blockIdx.y, i = blockIdx.z;
    const int32_t G = a.group, BS = a.block_size;
    const int32_t q0 = a.query_start[i], L = a.query_start[i + 1] - q0;
    const int32_t T = clamp_len(a, a.seq_lens[i]);
    if (L > T) {
        if (tid == 0 && tile == 0 && g == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int32_t tpt = C::kRows / G;                     // tokens per tile
    const int32_t tok0 = tile * tpt;
    if (L <= 0 || tok0 >= L) return;
    const int32_t ntok = min(tpt, L - tok0);
    const int32_t pos0 = T - L + tok0;
    const int32_t nkeys = pos0 + ntok;
    const int32_t nb = (nkeys + C::kKeys - 1) / C::kKeys;  // key blocks
    const int32_t nblk = (nkeys + BS - 1) / BS;            // paged blocks
    const int32_t cpb = BS >= C::kChunk ? BS / C::kChunk : 1;
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;

    // this thread's row
    const int32_t tok = tid / G, head = tid - (tid / G) * G;
    const bool row_ok = tok < ntok;
    const int32_t pos = pos0 + (row_ok ? tok : ntok - 1);
    const int64_t row_elem = ((int64_t)(q0 + tok0 + tok) * a.num_q_heads + g * G + head) * D;

    if (warp == 0) tmem_alloc(smem_u32(tslot), C::kTmemCols);

    // Q row -> shared memory, 128-byte swizzle per 64-column slice
    {
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row_ok) v = *reinterpret_cast<const uint4*>(q + row_elem + c * 8);
            const int h = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4*>(sm + C::kQOff + h * C::kQSlice + tid * 128 +
                                      ((cc ^ (tid & 7)) << 4)) = v;
        }
    }
    fence_proxy_async_smem();

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
    // paged blocks touched by key block kb
    auto first_blk = [&](int32_t kb) { return (kb * C::kKeys) / BS; };
    auto last_blk = [&](int32_t kb) { return (min(kb * C::kKeys + C::kKeys, nkeys) - 1) / BS; };

    fill_window(0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t s_tmem = tmem;
    const uint32_t o_tmem = tmem + C::kOCol;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    const uint64_t policy = l2_policy_evict_first();
    // thread 0: TMA copies of key block kb into stage kb % kStages
    auto issue = [&](int32_t kb) {
        const int32_t st = kb % C::kStages;
        const uint32_t bar = smem_u32(&bars[st]);
        const int32_t w0 = s_win0;
        bool ok = true;
        for (int32_t b = first_blk(kb); b <= last_blk(kb); ++b) ok = ok && win[b - w0] >= 0;
        s_stage_ok[st] = ok;
        if (!ok) {
            mbar_arrive(bar);
            return;
        }
        const uint32_t kdst = sm_u + C::kStageOff + st * C::kStageBytes;
        const uint32_t vdst = kdst + C::kTile;
        // bytes this block's copies deliver: per 16-key chunk, K and V, every
        // 64-column slice, 16 rows (or 8 per 8-token block that exists)
        uint32_t bytes = 0;
        for (int j = 0; j < C::kKeys / C::kChunk; ++j) {
            const int32_t key0 = kb * C::kKeys + j * C::kChunk;
            if (key0 >= nkeys) break;
            const int32_t halves = BS >= C::kChunk ? 2 : ((key0 / BS) + 1 < nblk ? 2 : 1);
            bytes += (uint32_t)halves * (C::kBox / 2) * C::kHalves * 2;
        }
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, bytes);
        for (int j = 0; j < C::kKeys / C::kChunk; ++j) {
            const int32_t key0 = kb * C::kKeys + j * C::kChunk;
            if (key0 >= nkeys) break;
            const int32_t c = key0 / C::kChunk;              // chunk index in the sequence
            if (BS >= C::kChunk) {
                const int32_t blk = c / cpb;
                const int32_t y = (c - blk * cpb) * C::kChunk;
                const int32_t z = win[blk - w0] * a.num_kv_heads + g;
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {
                    tma_load_3d_hint(kdst + h * C::kSlice + j * C::kBox, &tmap_k, h * 64, y, z,
                                     bar, policy);
                    tma_load_3d_hint(vdst + h * C::kSlice + j * C::kBox, &tmap_v, h * 64, y, z,
                                     bar, policy);
                }
            } else {
                const int32_t b0 = 2 * c;
                for (int half = 0; half < 2 && b0 + half < nblk; ++half) {
                    const int32_t z = win[b0 + half - w0] * a.num_kv_heads + g;
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h) {
                        tma_load_3d_hint(kdst + h * C::kSlice + j * C::kBox + half * 1024,
                                         &tmap_k, h * 64, 0, z, bar, policy);
                        tma_load_3d_hint(vdst + h * C::kSlice + j * C::kBox + half * 1024,
                                         &tmap_v, h * 64, 0, z, bar, policy);
                    }
                }
            }
        }
    };
    // thread 0: S = Q K^T for key block kb (its stage has landed)
    constexpr uint32_t kIdescS = umma_idesc_bf16(128, C::kKeys, 0);
    constexpr uint32_t kIdescO = umma_idesc_bf16(128, 64, 1);
    auto issue_s = [&](int32_t kb) {   // thread 0; S buffer kb & 1
        const int32_t st = kb % C::kStages;
        const uint32_t bar = bar_s0 + 8 * (kb & 1);
        if (!s_stage_ok[st]) {
            mbar_arrive(bar);
            return;
        }
        const uint32_t kbase = sm_u + C::kStageOff + st * C::kStageBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t ad =
                umma_sdesc(sm_u + C::kQOff + (ks >> 2) * C::kQSlice + (ks & 3) * 32, 16, 1024, 2);
            const uint64_t bd = umma_sdesc(kbase + (ks >> 2) * C::kSlice + (ks & 3) * 32, 16,
                                           1024, 2);
            umma_bf16(s_tmem + (kb & 1) * C::kKeys, ad, bd, kIdescS, ks > 0);
        }
        umma_commit(bar);
    };

    bool failed = false;
    bool o_init = false;                               // thread 0: O written at least once
    bool t0_fail = false;                              // thread 0: a stage copy never landed
    if (tid == 0) {
        for (int32_t kb = 0; kb < min(nb, C::kStages); ++kb) issue(kb);
        if (!mbar_wait_bounded(smem_u32(&bars[0]), 0, kWaitLimitCycles)) {
            t0_fail = true;
            mbar_arrive(bar_s0);
        } else {
            tc_fence_after();
            issue_s(0);
        }
    }

    // m_ref: the reference maximum P is taken against.  It moves only when a
    // row's maximum exceeds it by more than 8 (base 2), so O is rescaled
    // rarely; P stays <= 2^8 and O / l does not depend on the reference.
    constexpr float kRescaleSlack = 8.f;
    float m_ref = -INFINITY, l = 0.f;
    for (int32_t kb = 0; kb < nb; ++kb) {
        const int32_t st = kb % C::kStages;
        const uint32_t bar_s = bar_s0 + 8 * (kb & 1);
        const bool s_ready =
            t0_fail ? false : mbar_wait_bounded(bar_s, (kb >> 1) & 1, kWaitLimitCycles);
        if (__syncthreads_or(!s_ready)) {
            failed = true;
            break;
        }
        tc_fence_after();
        // start S of the next block now: it runs while this block's softmax does
        if (tid == 0 && kb + 1 < nb) {
            const int32_t st1 = (kb + 1) % C::kStages;
            if (!mbar_wait_bounded(smem_u32(&bars[st1]), ((kb + 1) / C::kStages) & 1,
                                   kWaitLimitCycles)) {
                t0_fail = true;                // reported at the next S barrier
                mbar_arrive(bar_s0 + 8 * ((kb + 1) & 1));
            } else {
                tc_fence_after();
                issue_s(kb + 1);
            }
        }
        const bool ok = s_stage_ok[st];
        float sv[32];
        if (ok) tmem_ld32(s_tmem + (kb & 1) * C::kKeys + lane_base, sv);
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int32_t key = kb * C::kKeys + j;
            sv[j] = (ok && key <= pos) ? sv[j] * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, sv[j]);
        }
        const bool raise = mx > m_ref + kRescaleSlack || (m_ref == -INFINITY && mx > -INFINITY);
        const float m_new = raise ? mx : m_ref;
        const float alpha = raise ? exp2f(m_ref - m_new) : 1.f;   // 0 when m_ref = -inf
        float rs = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            sv[j] = m_new == -INFINITY ? 0.f : exp2f(sv[j] - m_new);
            rs += sv[j];
        }
        l = l * alpha + rs;
        m_ref = m_new;
        // the previous P V must be done before O is rescaled or P is rewritten
        if (kb > 0) {
            if (__syncthreads_or(!mbar_wait_bounded(bar_o, (kb - 1) & 1, kWaitLimitCycles))) {
                failed = true;
                break;
            }
            tc_fence_after();
            if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float ov[32];
                    tmem_ld32(o_tmem + lane_base + c * 32, ov);
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] *= alpha;
                    tmem_st32(o_tmem + lane_base + c * 32, ov);
                }
            }
        }
        // P row -> shared memory: K-major core matrices (8 rows x 16 bytes),
        // 8-row groups 512 bytes apart, key chunks 128 bytes apart
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
            uint4 v;
            v.x = pack_bf16x2(sv[kc * 8 + 0], sv[kc * 8 + 1]);
            v.y = pack_bf16x2(sv[kc * 8 + 2], sv[kc * 8 + 3]);
            v.z = pack_bf16x2(sv[kc * 8 + 4], sv[kc * 8 + 5]);
            v.w = pack_bf16x2(sv[kc * 8 + 6], sv[kc * 8 + 7]);
            *reinterpret_cast<uint4*>(sm + C::kPOff + (tid >> 3) * 512 + kc * 128 + (tid & 7) * 16) = v;
        }
        // keys past the last position in the final block: clear their V rows
        const int32_t nvalid = nkeys - kb * C::kKeys;
        if (nvalid < C::kKeys) {
            uint8_t* vt = sm + C::kStageOff + st * C::kStageBytes + C::kTile;
            const int32_t pieces = (C::kKeys - nvalid) * 8;
            for (int32_t x = tid; x < C::kHalves * pieces; x += C::kThreads) {
                const int32_t h = x / pieces, r = x - h * pieces;
                *reinterpret_cast<uint4*>(vt + h * C::kSlice + nvalid * 128 + r * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            if (ok) {
                const uint32_t vbase = sm_u + C::kStageOff + st * C::kStageBytes + C::kTile;
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
                    for (int ks = 0; ks < C::kKeys / 16; ++ks) {
                        const uint64_t ad = umma_sdesc(sm_u + C::kPOff + ks * 256, 128, 512, 0);
                        const uint64_t bd = umma_sdesc(vbase + h * C::kSlice + ks * 2048, 16,
                                                       1024, 2);
                        umma_bf16(o_tmem + h * 64, ad, bd, kIdescO, (o_init || ks > 0) ? 1u : 0u);
                    }
                o_init = true;
                umma_commit(bar_o);
            } else {
                mbar_arrive(bar_o);
            }
        }
        // refill the stage of block kb - 1 (its S and P V have completed),
        // sliding the block-id window first when needed (uniform branch)
        const int32_t nxt = kb - 1 + C::kStages;
        if (kb >= 1 && nxt < nb) {
            if (last_blk(nxt) >= s_win0 + C::kWindow) {
                __syncthreads();
                fill_window(first_blk(nxt));
                __syncthreads();
            }
            if (tid == 0) issue(nxt);
        }
    }

    // last P V, then the epilogue
    bool o_ready = !failed;
    if (!failed && nb > 0)
        o_ready = mbar_wait_bounded(bar_o, (nb - 1) & 1, kWaitLimitCycles);
    if (__syncthreads_or(!o_ready)) failed = true;
    tc_fence_after();
    if (failed) {
        if (tid == 0) {
            // every MMA issued so far must finish before tensor memory is freed
            umma_commit(bar_fin);
            mbar_wait_bounded(bar_fin, 0, kWaitLimitCycles);
            raise_error(PA_DEVERR_TIMEOUT);
        }
        __syncthreads();
    } else {
        griddep_launch_dependents();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tmem_ld32(o_tmem + lane_base + c * 32, ov);
            if (row_ok) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v;
                    v.x = pack_bf16x2(ov[q4 * 8 + 0] * inv, ov[q4 * 8 + 1] * inv);
                    v.y = pack_bf16x2(ov[q4 * 8 + 2] * inv, ov[q4 * 8 + 3] * inv);
                    v.z = pack_bf16x2(ov[q4 * 8 + 4] * inv, ov[q4 * 8 + 5] * inv);
                    v.w = pack_bf16x2(ov[q4 * 8 + 6] * inv, ov[q4 * 8 + 7] * inv);
                    *reinterpret_cast<uint4*>(out + row_elem + c * 32 + q4 * 8) = v;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace pa
