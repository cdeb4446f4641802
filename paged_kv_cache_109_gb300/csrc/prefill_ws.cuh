// prefill_ws.cuh -- multi-query (chunked prefill) paged attention on the
// 5th-generation tensor cores (tcgen05, tensor-memory accumulators), bf16,
// with warp-specialised roles.
//
// Definition: sequence i's packed query rows are its last L_i positions; the
// row at position p attends to keys 0..p of the sequence through its block
// table ("vLLM source walkthrough: PagedAttention and Continuous Batching"
// §2.8; "vLLM PagedAttention: from memory fragmentation to slot mapping" §6).
//
// One CTA per (pair of query tiles, kv head g, sequence i).  A tile is 128
// MMA rows = (query token, query head of the group) pairs, head fastest, so
// it holds 128/G tokens; the CTA's two tiles are consecutive.  Both tiles
// share each key block, so K and V cross shared memory once per 256 rows.
//
//   warps 0-3  softmax of tile 0 (thread t owns tensor-memory lane t)
//   warps 4-7  softmax of tile 1
//   warp 8     producer: block-table lookups and TMA copies of K and V blocks
//              (KEYS keys each) into a ring of shared-memory slots
//   warp 9     MMA issue, fp32 accumulators in tensor memory:
//                S_t  = Q_t K^T   M128 x N KEYS, A and B from shared memory
//                O_t += P_t V     M128 x N D, A = P_t from tensor memory
//
// Tensor memory per tile: S_t (KEYS fp32 columns) and O_t (D columns).  P is
// taken as two bf16 parts, P = hi + lo (lo: the rounding error of hi, rounded
// again), so P V keeps about 16 significant bits of each weight instead of
// the 8 of one bf16 operand.  The softmax takes S_t one 64-key half at a time;
// once a half's 64 columns are in registers, its hi parts (bf16 pairs) go to
// the first 32 of them and its lo parts to the other 32, and the half is
// published.  Per key block kb the MMA warp issues, for t = 0, 1: O_t +=
// hi V + lo V for keys 0-63 of block kb - 1 as soon as that half is published
// (while the softmax computes keys 64-127), then the same for keys 64-127,
// then S_t(kb) into the same columns (tcgen05 MMAs of one thread run in issue
// order, so P_t is read before it is overwritten).  Each
// softmax warpgroup overlaps the other tile's tensor-core work, and with P
// off shared memory the K/V ring holds enough blocks to hide the copies'
// latency.
//
// Softmax per row and 64-key half: load S (tcgen05.ld), mask keys past the
// row's position (diagonal blocks only), take the half's maximum, p = 2^(s c
// - m) with c = scale log2(e) and a lazily moved reference maximum m (it
// moves only when the maximum exceeds it by more than 8, so O is rescaled
// rarely, p <= 2^8 and O / l does not depend on m), accumulate l (from the
// fp32 p), store hi and lo.  O is divided by l at the end.
//
// Synchronisation is by mbarriers only; every wait is bounded, and a timeout
// raises PA_DEVERR_TIMEOUT and ends the role's work (the others then time
// out too) without leaving copies or MMAs in flight past the CTA's end.
#pragma once

#include <type_traits>

#include "prefill_args.cuh"

namespace pa {

template <int D, int KEYS>
struct PrefillWsCfg {
    static constexpr int kProducers = PA_PREFILL_PRODUCERS;   // copy-issuing warps
    static constexpr int kThreads = 32 * (9 + kProducers);
    static constexpr int kSoftmaxWarps = 8;
    static constexpr int kProducerWarp = 8;               // and warps 10, 11, ...
    static constexpr int kMmaWarp = 9;
    static constexpr int kTiles = 2;
    static constexpr int kRows = 128;                     // rows per tile = tensor-memory lanes
    static constexpr int kKeys = KEYS;                    // N of S, K of P V
    static constexpr int kHalves = D / 64;                // 64-column (128-byte) slices
    static constexpr int kSlice = kKeys * 128;            // one block, one slice
    static constexpr int kItem = kHalves * kSlice;        // K or V of one block
    static constexpr int kQSlice = kRows * 128;
    static constexpr int kQTile = kHalves * kQSlice;
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = kTiles * kQTile;
    static constexpr int kSmemMax = 232448;               // dynamic shared memory per CTA
    static constexpr int kSlots = (kSmemMax - 2048 - kSlotOff) / kItem;
    static constexpr int kBarOff = kSlotOff + kSlots * kItem;
    // K/V full, K/V empty; per tile S full, P half 0, P full, O half 0, O done; final
    static constexpr int kBars = 2 * kSlots + 11;
    static constexpr int kTslotOff = kBarOff + 8 * kBars;
    static size_t smem_bytes() { return 1024 + kTslotOff + 16; }
    static constexpr uint32_t kTmemCols = 512;            // per tile: S (and P) at +0, O at +128
    static constexpr uint32_t kTileCols = 256;
    static constexpr uint32_t kOCol = 128;
    static_assert(D == 64 || D == 128, "tile width");
    static_assert(KEYS == 128, "key block: two 64-key halves");
    static_assert(kSlots >= 4, "ring");
};

template <int D, int KEYS>
__global__ void __launch_bounds__(PrefillWsCfg<D, KEYS>::kThreads, 1)
prefill_ws_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    using C = PrefillWsCfg<D, KEYS>;
    extern __shared__ uint8_t sm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sm_u = smem_u32(sm);
    const uint32_t bar0 = sm_u + C::kBarOff;
    auto kv_full = [&](int32_t s) { return bar0 + 8u * s; };
    auto kv_empty = [&](int32_t s) { return bar0 + 8u * (C::kSlots + s); };
    auto s_full = [&](int32_t t) { return bar0 + 8u * (2 * C::kSlots + t); };
    auto p_full = [&](int32_t t) { return bar0 + 8u * (2 * C::kSlots + 2 + t); };
    auto o_done = [&](int32_t t) { return bar0 + 8u * (2 * C::kSlots + 4 + t); };
    auto p_half = [&](int32_t t) { return bar0 + 8u * (2 * C::kSlots + 6 + t); };
    auto o_half = [&](int32_t t) { return bar0 + 8u * (2 * C::kSlots + 8 + t); };
    const uint32_t bar_fin = bar0 + 8u * (2 * C::kSlots + 10);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::kTslotOff);

    const int32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int32_t s = 0; s < C::kSlots; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int32_t t = 0; t < C::kTiles; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 4);                      // one arrival per softmax warp
            mbar_init(o_done(t), 1);
            mbar_init(p_half(t), 4);
            mbar_init(o_half(t), 1);
        }
        mbar_init(bar_fin, 1);
        mbar_fence_init();
    }
    if (warp == C::kProducerWarp && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    griddep_wait();

    const int32_t cta = gridDim.x - 1 - blockIdx.x;       // latest (longest) tiles first
    const int32_t g = blockIdx.y, i = blockIdx.z;
    const int32_t G = a.group, BS = a.block_size;
    const int32_t q0 = a.query_start[i], L = a.query_start[i + 1] - q0;
    const int32_t T = clamp_len(a, a.seq_lens[i]);
    if (L > T) {
        if (tid == 0 && cta == 0 && g == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int32_t tpt = C::kRows / G;                     // tokens per tile
    const int32_t tok0 = cta * C::kTiles * tpt;
    if (L <= 0 || tok0 >= L) return;
    const int32_t ntok = min(C::kTiles * tpt, L - tok0);
    const int32_t ntiles = ntok > tpt ? 2 : 1;
    const int32_t pos0 = T - L + tok0;
    const int32_t nkeys = pos0 + ntok;
    const int32_t nb = (nkeys + C::kKeys - 1) / C::kKeys;

    if (warp == C::kMmaWarp) tmem_alloc(smem_u32(tslot), C::kTmemCols);

    // softmax threads: row r of tile w
    const int32_t w = warp >> 2, r = tid & (C::kRows - 1);
    const int32_t tok = w * tpt + r / G, head = r - (r / G) * G;
    const bool softmax = warp < C::kSoftmaxWarps && w < ntiles;
    // rows past tpt * G (G not dividing 128) carry nothing: no Q, no output
    const bool row_ok = softmax && r < tpt * G && tok < ntok;
    const int32_t pos = pos0 + min(tok, ntok - 1);
    // the head dim; the tile is D columns (head dims 16-48 in a 64-column
    // tile, 80-112 in a 128-column one: the columns past hd are zeros in Q,
    // K and V and never stored)
    const int32_t hd = a.head_dim;
    const int64_t row_elem = ((int64_t)(q0 + tok0 + tok) * a.num_q_heads + g * G + head) * hd;
    if (softmax) {
        // Q row -> shared memory, 128-byte swizzle per 64-column slice
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
        for (int32_t c = 0; c < D / 8; ++c) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row_ok && c * 8 < hd) v = *reinterpret_cast<const uint4*>(q + row_elem + c * 8);
            const int32_t h = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4*>(sm + C::kQOff + w * C::kQTile + h * C::kQSlice + r * 128 +
                                      ((cc ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // a bounded wait whose outcome is the same in every lane of the warp
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kWaitLimitCycles)) != 0;
    };

    if (warp == C::kProducerWarp || warp > C::kMmaWarp) {
        // ---- producers -----------------------------------------------------
        // kProducers warps share the ring round-robin (item j is issued by
        // producer j % kProducers), so several warps' copies are in flight.
        const int32_t parity = warp == C::kProducerWarp ? 0 : warp - C::kMmaWarp;
        // Ring items in the order the MMA warp consumes them: K(0), then per
        // block kb: K(kb + 1), V(kb); so K runs a block ahead of V.  Lane j
        // copies the j-th box of a block; its block-table entry is read two
        // blocks ahead of use, so the lookup latency overlaps the waits.
        const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;
        const int32_t sub = BS >= 16 ? 16 : BS;           // rows per TMA box
        const int32_t nsub = C::kKeys / sub;
        const uint32_t box_bytes = (uint32_t)sub * 128u;
        auto lookup = [&](int32_t kb) {                    // raw table entry of lane's box
            const int32_t key0 = kb * C::kKeys + lane * sub;
            return (kb < nb && lane < nsub && key0 < nkeys) ? table[key0 / BS] : 0;
        };
        struct Box {
            bool has;
            int32_t y, z;
            uint32_t bytes;
        };
        auto decode = [&](int32_t kb, int32_t id) {
            Box bx{false, 0, -1, 0u};
            const int32_t key0 = kb * C::kKeys + lane * sub;
            bx.has = lane < nsub && key0 < nkeys;
            if (bx.has) {
                bx.y = key0 - (key0 / BS) * BS;
                if (id < 0 || id >= a.num_blocks)
                    raise_error(PA_DEVERR_TABLE_ENTRY);       // z = -1: the box reads zeros
                else
                    bx.z = id * a.num_kv_heads + g;
            }
            bx.bytes = __popc(__ballot_sync(0xffffffffu, bx.has)) * box_bytes * C::kHalves;
            return bx;
        };
        int32_t it = 0;                                   // ring items issued
        bool ok = true;
        auto issue = [&](const Box& bx, bool is_v) {
            if (it % C::kProducers != parity) {
                ++it;
                return;
            }
            const int32_t s = it % C::kSlots;
            if (it >= C::kSlots && !warp_wait(kv_empty(s), ((it / C::kSlots) - 1) & 1)) {
                ok = false;
                return;
            }
            if (lane == 0) mbar_arrive_expect_tx(kv_full(s), bx.bytes);
            __syncwarp();
            if (bx.has) {
                const uint32_t dst = sm_u + C::kSlotOff + s * C::kItem + lane * box_bytes;
                const void* map =
                    is_v ? static_cast<const void*>(&tmap_v) : static_cast<const void*>(&tmap_k);
#pragma unroll
                for (int32_t h = 0; h < C::kHalves; ++h)
                    tma_load_3d(dst + h * C::kSlice, map, h * 64, bx.y, bx.z, kv_full(s));
            }
            ++it;
        };
        Box cur = decode(0, lookup(0));
        int32_t raw_next = lookup(1);
        issue(cur, false);                                // K(0)
        for (int32_t kb = 0; kb < nb && ok; ++kb) {
            const int32_t raw_after = lookup(kb + 2);
            Box nxt{};
            if (kb + 1 < nb) {
                nxt = decode(kb + 1, raw_next);
                issue(nxt, false);                        // K(kb + 1)
            }
            if (ok) issue(cur, true);                     // V(kb)
            cur = nxt;
            raw_next = raw_after;
        }
        // the last copy into each slot has landed before the CTA may end
        for (int32_t j = max(0, it - C::kSlots); j < it; ++j)
            if (j % C::kProducers == parity)
                mbar_wait_bounded(kv_full(j % C::kSlots), (j / C::kSlots) & 1, kWaitLimitCycles);
        if (!ok && lane == 0) raise_error(PA_DEVERR_TIMEOUT);
    } else if (warp == C::kMmaWarp) {
        // ---- MMA issue -----------------------------------------------------
        constexpr uint32_t kIdS = umma_idesc_bf16(128, C::kKeys, 0);
        // P V produces the head dim's columns only (N = hd, a multiple of 16):
        // in the 128-column tile of head dims 80-112 the rest of V is zeros
        const uint32_t kIdO = umma_idesc_bf16(128, hd, 1);
        // Descriptors of step 0; a step adds its byte offset / 16 to the start
        // address field (addresses stay below 2^18, so the field never carries).
        uint64_t qdesc[C::kTiles];
#pragma unroll
        for (int32_t t = 0; t < C::kTiles; ++t)
            qdesc[t] = umma_sdesc(sm_u + C::kQOff + t * C::kQTile, 16, 1024, 2);
        const bool leader = elect_one();
        bool ok = true;
        for (int32_t kb = 0; kb <= nb && ok; ++kb) {
            // ring items: K(0) = 0, K(kb) = 2 kb - 1; V(kb) = 2 kb + 2, or 2 kb + 1
            // for the last block (no K(kb + 1) before it)
            const int32_t kit = kb == 0 ? 0 : 2 * kb - 1;
            const int32_t vit = kb == 0 ? -1 : (kb < nb ? 2 * kb : 2 * kb - 1);   // V(kb - 1)
            const int32_t ks = kit % C::kSlots, vs = (vit + C::kSlots) % C::kSlots;
            // K: K-major, 128-byte swizzle; V: MN-major, 64-column atoms kSlice
            // bytes apart (LBO)
            const uint64_t kdesc = umma_sdesc(sm_u + C::kSlotOff + ks * C::kItem, 16, 1024, 2);
            const uint64_t vdesc =
                umma_sdesc(sm_u + C::kSlotOff + vs * C::kItem, C::kSlice, 1024, 2);
            if (kb < nb) ok = warp_wait(kv_full(ks), (kit / C::kSlots) & 1);
            if (ok && kb > 0) {
                ok = warp_wait(kv_full(vs), (vit / C::kSlots) & 1);
                const int32_t nvalid = nkeys - (kb - 1) * C::kKeys;
                if (ok && kb == nb && nvalid < C::kKeys) {
                    // V rows past the last key may hold anything (NaN): clear them
                    uint8_t* vt = sm + C::kSlotOff + vs * C::kItem;
                    const int32_t pieces = (C::kKeys - nvalid) * 8;
                    for (int32_t x = lane; x < C::kHalves * pieces; x += 32) {
                        const int32_t h = x / pieces, rr = x - h * pieces;
                        *reinterpret_cast<uint4*>(vt + h * C::kSlice + nvalid * 128 + rr * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
            }
            for (int32_t t = 0; t < ntiles && ok; ++t) {
                const uint32_t s_t = tmem + t * C::kTileCols;
                if (kb > 0) {
                    // O_t += P_t(kb - 1) V(kb - 1) in two halves: keys 0-63 as soon
                    // as softmax t publishes them, keys 64-127 after; each half
                    // as hi V + lo V
#pragma unroll
                    for (int32_t hf = 0; hf < 2; ++hf) {
                        if (!warp_wait(hf ? p_full(t) : p_half(t), (kb - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (leader) {
                            // half hf: hi at columns 64 hf .. 64 hf + 31,
                            // lo at the next 32; 16 keys = 8 columns per step
#pragma unroll
                            for (int32_t k = 0; k < 4; ++k)
                                umma_bf16_ts(s_t + C::kOCol, s_t + hf * 64 + k * 8,
                                             vdesc + (uint64_t)((hf * 4 + k) * 128), kIdO,
                                             (kb > 1 || hf > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                            for (int32_t k = 0; k < 4; ++k)
                                umma_bf16_ts(s_t + C::kOCol, s_t + hf * 64 + 32 + k * 8,
                                             vdesc + (uint64_t)((hf * 4 + k) * 128), kIdO, 1u);
                            umma_commit(hf ? o_done(t) : o_half(t));
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                }
                if (kb < nb && leader) {
                    // S_t(kb) = Q_t K(kb)^T over the columns P_t(kb - 1) occupied,
                    // k-steps of the head dim only
#pragma unroll
                    for (int32_t k = 0; k < D / 16; ++k) {
                        if (k < hd / 16)
                            umma_bf16(s_t,
                                      qdesc[t] + (uint64_t)((k >> 2) * (C::kQSlice >> 4) + (k & 3) * 2),
                                      kdesc + (uint64_t)((k >> 2) * (C::kSlice >> 4) + (k & 3) * 2),
                                      kIdS, k > 0 ? 1u : 0u);
                    }
                    umma_commit(s_full(t));
                }
                __syncwarp();
            }
            if (ok && leader) {
                if (kb < nb) umma_commit(kv_empty(ks));
                if (kb > 0) umma_commit(kv_empty(vs));
            }
            __syncwarp();
        }
        // every MMA issued has finished before tensor memory is released
        if (leader) umma_commit(bar_fin);
        __syncwarp();
        mbar_wait_bounded(bar_fin, 0, kWaitLimitCycles);
        if (!ok && lane == 0) raise_error(PA_DEVERR_TIMEOUT);
    } else if (softmax) {
        // ---- softmax of tile w, row r --------------------------------------
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + w * C::kTileCols + lane_base;
        const uint32_t o_tm = s_tm + C::kOCol;
        const float c = a.scale_log2;                     // >= 0 on this path
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int32_t kb = 0; kb < nb; ++kb) {
            if (!warp_wait(s_full(w), kb & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int32_t key0 = kb * C::kKeys;
            const bool full = key0 + C::kKeys - 1 <= pos;
            // Each 64-key half of S: load it, take its maximum, move this row's
            // reference m_ref if that maximum exceeds it by more than 8, p =
            // 2^(s c - m_ref) (packed fp32 FMA and add), P as hi + lo -> tensor
            // memory over the half's own 64 columns of S_t (read by then;
            // P_t(kb - 1) V(kb - 1) ran before S_t(kb)), rescale O
            // if the reference moved (once the P V it holds has finished), and
            // publish the half: the MMA warp starts O += P V on keys 0-63 while
            // keys 64-127 are still being computed.
            const float2 c2 = make_float2(c, c);
            auto block = [&](auto masked) -> bool {
                constexpr bool kMasked = decltype(masked)::value;
                uint32_t sr[2][32];
                tmem_ld32_async(s_tm, sr[0]);
                tmem_ld32_async(s_tm + 32, sr[1]);
                tmem_wait_ld();
                tmem_regs_ready(sr[0]);
                tmem_regs_ready(sr[1]);
#pragma unroll
                for (int32_t hh = 0; hh < 2; ++hh) {
                    if constexpr (kMasked) {
#pragma unroll
                        for (int32_t j = 0; j < 64; ++j)
                            if (key0 + hh * 64 + j > pos) sr[j >> 5][j & 31] = __float_as_uint(-INFINITY);
                    }
                    float mp[4];
#pragma unroll
                    for (int32_t u = 0; u < 4; ++u) mp[u] = -INFINITY;
#pragma unroll
                    for (int32_t jj = 0; jj < 32; ++jj)
                        mp[jj & 3] = fmax3(mp[jj & 3], __uint_as_float(sr[(2 * jj) >> 5][(2 * jj) & 31]),
                                           __uint_as_float(sr[(2 * jj + 1) >> 5][(2 * jj + 1) & 31]));
                    const float mraw = fmaxf(fmax3(mp[0], mp[1], mp[2]), mp[3]);
                    const float mx = mraw == -INFINITY ? -INFINITY : mraw * c;
                    const bool up = mx > m_ref + 8.f;
                    const float a = up ? ex2_approx(m_ref - mx) : 1.f;   // 0 when m_ref = -inf
                    if (up) m_ref = mx;
                    l *= a;
                    const float ref = m_ref == -INFINITY ? 0.f : m_ref;
                    const float2 nm2 = make_float2(-ref, -ref);
                    float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    uint32_t pk[32], plo[32];                 // hi and lo parts of P
#pragma unroll
                    for (int32_t jj = 0; jj < 32; ++jj) {
                        const int32_t j = 2 * jj;
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[j >> 5][j & 31]),
                                                                __uint_as_float(sr[(j + 1) >> 5][(j + 1) & 31])),
                                                    c2, nm2);
                        float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        if constexpr (kMasked) {             // c = 0: -inf * 0 is NaN
                            pp.x = key0 + hh * 64 + j <= pos ? pp.x : 0.f;
                            pp.y = key0 + hh * 64 + j + 1 <= pos ? pp.y : 0.f;
                        }
                        rs[jj & 1] = __fadd2_rn(rs[jj & 1], pp);
                        split_bf16x2(pp.x, pp.y, pk[jj], plo[jj]);
                    }
                    // this half's 64 columns of S are in registers: hi and lo
                    // take them
                    tmem_st32_async(s_tm + hh * 64, pk);
                    tmem_st32_async(s_tm + hh * 64 + 32, plo);
                    l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
                    // the second half's scores load while this half is published
                    if (hh == 0) {
                        tmem_ld32_async(s_tm + 64, sr[0]);
                        tmem_ld32_async(s_tm + 96, sr[1]);
                    }
                    // O holds the P V of every earlier half: rescale it once that
                    // has finished, before this half is published (nothing to
                    // rescale before the first half)
                    if ((kb > 0 || hh > 0) && __any_sync(0xffffffffu, up)) {
                        const bool waited = hh == 0 ? warp_wait(o_done(w), (kb - 1) & 1)
                                                    : warp_wait(o_half(w), kb & 1);
                        if (!waited) return false;
                        tc_fence_after();
#pragma unroll
                        for (int32_t cc = 0; cc < D / 32; ++cc) {
                            float ov[32];
                            tmem_ld32(o_tm + cc * 32, ov);
#pragma unroll
                            for (int32_t j = 0; j < 32; ++j) ov[j] *= a;
                            tmem_st32(o_tm + cc * 32, ov);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(hh == 0 ? p_half(w) : p_full(w));
                    if (hh == 0) {
                        tmem_wait_ld();
                        tmem_regs_ready(sr[0]);
                        tmem_regs_ready(sr[1]);
                    }
                }
                return true;
            };
            // the version is chosen per warp (the tcgen05 accesses inside are
            // warp-collective): unmasked only when every row sees the whole block
            const bool warp_full = __all_sync(0xffffffffu, full) != 0;
            ok = warp_full ? block(std::false_type{}) : block(std::true_type{});
            if (!ok) break;
        }
        if (ok) ok = warp_wait(o_done(w), (nb - 1) & 1);
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
            for (int32_t cc = 0; cc < D / 32; ++cc) {
                float ov[32];
                tmem_ld32(o_tm + cc * 32, ov);
                if (row_ok) {
#pragma unroll
                    for (int32_t q4 = 0; q4 < 4; ++q4) {
                        if (cc * 32 + q4 * 8 >= hd) break;   // past the head dim
                        uint4 v;
                        v.x = pack_bf16x2(ov[q4 * 8 + 0] * inv, ov[q4 * 8 + 1] * inv);
                        v.y = pack_bf16x2(ov[q4 * 8 + 2] * inv, ov[q4 * 8 + 3] * inv);
                        v.z = pack_bf16x2(ov[q4 * 8 + 4] * inv, ov[q4 * 8 + 5] * inv);
                        v.w = pack_bf16x2(ov[q4 * 8 + 6] * inv, ov[q4 * 8 + 7] * inv);
                        *reinterpret_cast<uint4*>(out + row_elem + cc * 32 + q4 * 8) = v;
                    }
                }
            }
        } else if (lane == 0) {
            raise_error(PA_DEVERR_TIMEOUT);
        }
    }
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace pa
