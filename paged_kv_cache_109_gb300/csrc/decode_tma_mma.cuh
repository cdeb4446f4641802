// decode_tma_mma.cuh -- bf16 paged decode: TMA tile loads driven by the block
// table, tensor-core score and value contractions, online softmax.
//
// Work split.  One CTA per (partition p, kv head g, sequence i); four warps.
// The partition's block ids are read from the table once into shared memory.
// The partition's tokens are cut into 16-token chunks (a block of B tokens,
// B a multiple of 16, is B/16 chunks).  Warp w takes chunks w, w+4, w+8, ...
// and keeps a private ring of kStages shared-memory stages; one stage holds
// the K rows and the V rows of one chunk of one (physical block, kv head)
// tile, 16 x head_dim contiguous in the cache.  Lane 0 issues 3-D
// bulk-tensor copies (TMA, 128-byte swizzle) for the chunk kStages ahead,
// completion counted on the stage's mbarrier, so the table walk doubles as
// the prefetch schedule
// ("vLLM source walkthrough: PagedAttention and Continuous Batching" §1.8:
// block_table[block_idx] gives the physical block whose K/V the kernel loads;
// the kernel walks the table's blocks).
//
// Per chunk, with the G <= 16 query heads of the kv group as the 16 rows of
// an m16n8k16 tile (rows >= G are zero), the warp computes
//   S[16 x 16]  = Q[16 x D] . K_chunk^T         (ldmatrix from the swizzled tile)
//   online softmax on S in base 2 (scale * log2 e folded into one multiply):
//   m' = max(m, rowmax S), acc *= 2^(m - m'), P = 2^(S - m'), l = l 2^(m-m') + rowsum P
//   acc[16 x D] += P[16 x 16] . V_chunk           (P re-used from the S registers)
// so every K/V tile is read from HBM once for all heads of its group
// (the glossary page's expand_kv grouping: head h reads kv head h / G).
// Positions at or past T_i inside the last chunk are masked to -inf (nxmr.cn
// article §2.2: whole-block loads, padding masked).
//
// At the end the four warps' (m, l, acc) are combined through shared memory;
// a sequence that fits one partition writes its output, otherwise the
// partition's (acc, m, l) go to the workspace for merge_kernel.
#pragma once

#include <cuda.h>

#include "decode_generic.cuh"
#include "ptx.cuh"

namespace pa {

// Shared-memory ring per warp (bytes) and the CTAs per SM the launch bounds
// ask for.  Two 8 KiB stages per warp (D = 128) and three CTAs per SM keep
// 96-192 KiB of K/V in flight per SM, and one CTA's prologue or epilogue
// overlaps the others' streaming (measured best of 1-3 CTAs x 2-4 stages).
#ifndef PA_RING_BYTES_PER_WARP
#define PA_RING_BYTES_PER_WARP 16384
#endif
#ifndef PA_MIN_CTAS_PER_SM
#define PA_MIN_CTAS_PER_SM 3
#endif

template <int D, bool G16>
struct TmaMmaCfg {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kChunk = 16;                     // tokens per pipeline stage
    static constexpr int kBoxCols = 64;                   // 64 bf16 = 128 bytes (swizzle span)
    // head dims 16-48 and 80-112: the (last) box's columns past D arrive as zeros
    static constexpr int kBoxes = (D + kBoxCols - 1) / kBoxCols;
    static constexpr int kBoxBytes = kChunk * 128;        // 16 rows x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;  // 16 rows x kBoxes x 64 columns
    static constexpr int kStageBytes = 2 * kTileBytes;    // K chunk + V chunk
    static constexpr int kStagesRaw = PA_RING_BYTES_PER_WARP / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
    static constexpr int kRows = G16 ? 16 : 8;              // query-head rows carried
    static constexpr int kKSteps = D / 16;
    static constexpr int kDTiles = D / 8;
    static constexpr int kMaxTableSlice = 2048;            // block ids per partition
    static_assert(D % 16 == 0 && D <= 256, "tile shape");
    static_assert(kWarps * kRows * (D + 2) * 4 <= kRingBytes, "combine area");
    // dynamic shared bytes for a partition of part_tokens tokens
    static size_t smem_bytes(int32_t part_tokens, int32_t block_size) {
        const size_t ids =
            ((size_t)(part_tokens + block_size - 1) / block_size * 4 + 15) / 16 * 16;
        return 1024 + kRingBytes + 8 * kWarps * kStages + ids;
    }
    static size_t smem_bytes_max() { return smem_bytes(kMaxTableSlice, 1); }
};

// Head dim 256 holds a 256-column accumulator and 16 k-steps of Q in
// registers: one CTA per SM (up to 255 registers a thread), two 16 KiB
// stages per warp.
template <int D, bool G16, bool CAS>
__global__ void __launch_bounds__(128, D > 128 ? 1 : PA_MIN_CTAS_PER_SM)
decode_tma_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
    using C = TmaMmaCfg<D, G16>;
    extern __shared__ uint8_t sm_raw[];
    __shared__ int s_fail;
    // CAS (shared-prefix decode) only: per MMA row of a prefix CTA, its q (and
    // output) row, -1 for none, and the keys of the prefix it sees
    __shared__ int64_t s_qrow[CAS ? C::kRows : 1];
    __shared__ int32_t s_lim[CAS ? C::kRows : 1];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));

    // blockIdx.y = kv head g, sub-group sg: this CTA carries the group's
    // query heads sg * 16 .. sg * 16 + G - 1.  With CAS, blockIdx.z below
    // a.prefix_z is a prefix CTA: the shared leading blocks of one group of
    // sequences, its rows (member, query head) pairs; the other CTAs run
    // sequence blockIdx.z - a.prefix_z, a group member past its group's
    // shared blocks.
    const bool pre = CAS && (int32_t)blockIdx.z < a.prefix_z;
    const int32_t p = blockIdx.x, g = blockIdx.y / a.sub_groups;
    const int32_t i = CAS ? (int32_t)blockIdx.z - a.prefix_z : (int32_t)blockIdx.z;
    const int32_t sg = blockIdx.y - g * a.sub_groups;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t grp = lane >> 2, tig = lane & 3;
    const int32_t G = pre ? C::kRows : min(16, a.group - sg * 16);
    const int32_t BS = a.block_size;
    // B >= 16: a block is cpb = B/16 chunks.  B = 8: a chunk is two blocks,
    // loaded as two 8-row boxes (the 128-byte swizzle atom is 8 rows).
    const int32_t cpb = BS >= C::kChunk ? BS / C::kChunk : 1;
    const int32_t P = a.part_tokens;
    const int32_t t0 = p * P;
    const int64_t head0 = (int64_t)i * a.num_q_heads + (int64_t)g * a.group + sg * 16;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kRingBytes);
    int32_t* ids = reinterpret_cast<int32_t*>(bars + C::kWarps * C::kStages);

    // Barrier set-up reads no input, so it runs before waiting for the
    // previous kernel in the stream (programmatic dependent launch); every
    // input read comes after griddep_wait().
    if (tid == 0) {
        for (int s2 = 0; s2 < C::kWarps * C::kStages; ++s2) mbar_init(smem_u32(&bars[s2]), 1);
        mbar_fence_init();
        s_fail = 0;
    }
    if (tid == 32) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    griddep_wait();

    // Prologue.  Partition 0 of a sequence always has work (unless T = 0), so
    // its CTA issues the length, its slice of the block table (read
    // speculatively up to the partition's end, clamped to the row) and the
    // query fragments together: one memory round trip before the first tile
    // copy.  CTAs of later partitions are often empty (short sequences in a
    // batch sized by max_seq_len): they read the length first and leave at
    // once when there is nothing to do.
    // CAS: skip = tokens of the table row before this CTA's token 0 (a
    // member's shared blocks), slot0 = its partitions' first workspace slot
    // (after the group's prefix partitions), direct = may write out itself.
    int32_t T_raw, skip = 0, slot0 = 0;
    bool direct = true;
    const int32_t* row = nullptr;
    if (pre) {
        direct = false;
        const int32_t z = blockIdx.z, k = z / a.prefix_ztiles;
        const int32_t rt = (z - k * a.prefix_ztiles) * a.sub_groups + sg;   // row tile
        // member list [ms, ms + mc) inside members[0 .. member_start[num_groups])
        // and within the host bound; anything else is reported and skipped
        const int32_t total = a.member_start[a.num_groups];
        const int32_t ms = a.member_start[k], mc = a.member_start[k + 1] - ms;
        if (ms < 0 || mc < 0 || ms + mc > total || mc > a.max_group_size) {
            if (tid == 0) raise_error(PA_DEVERR_GROUP);
            return;
        }
        const int32_t pk = group_prefix_blocks(a, k) * BS;
        if (mc == 0 || t0 >= pk) return;
        if (tid < C::kRows) {
            // MMA row tid = pair rt * kRows + tid of the group's (member, head)
            // pairs, head fastest
            const int32_t u = rt * C::kRows + tid, mi = u / a.group, h = u - mi * a.group;
            int64_t qr = -1;
            int32_t lim = 0;
            if (mi < mc) {
                const int32_t sq = a.members[ms + mi];
                if (sq >= 0 && sq < a.num_seqs) {
                    qr = (int64_t)sq * a.num_q_heads + (int64_t)g * a.group + h;
                    lim = min(clamp_len(a, a.seq_lens[sq]), pk) - t0;   // keys of this partition
                } else {
                    raise_error(PA_DEVERR_GROUP);
                }
            }
            s_qrow[tid] = qr;
            s_lim[tid] = qr >= 0 ? max(0, min(lim, P)) : 0;
        }
        const int32_t first = a.members[ms];
        row = a.block_tables + (int64_t)(first >= 0 && first < a.num_seqs ? first : 0) *
                                   a.max_blocks;
        T_raw = pk;
        __syncthreads();
    } else {
        T_raw = a.seq_lens[i];
        if (CAS) {
            const int32_t k = seq_group_of(a, i);
            if (k >= 0) {
                const int32_t pk = group_prefix_blocks(a, k) * BS;
                direct = false;
                skip = pk;
                slot0 = (int32_t)(((int64_t)pk + P - 1) / P);
            }
        }
        if (p > 0 && T_raw - skip <= t0 && T_raw <= a.max_seq_len) return;
        row = a.block_tables + (int64_t)i * a.max_blocks;
    }
    const int32_t slice = max(0, min((P + BS - 1) / BS, a.max_blocks - (skip + t0) / BS));
    const int32_t* table = row + (skip + t0) / BS;
    constexpr int kIdsPerThread = (C::kMaxTableSlice + C::kThreads - 1) / C::kThreads;
    int32_t raw_ids[kIdsPerThread];
#pragma unroll
    for (int r = 0; r < kIdsPerThread; ++r) {
        const int32_t b = tid + r * C::kThreads;
        raw_ids[r] = b < slice ? table[b] : -1;
    }
    // Q fragments (A operand): rows = the group's query heads, k = head dim.
    uint32_t qa[C::kKSteps][4];
    {
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
        bool r0 = grp < G, r1 = G16 && (grp + 8) < G;
        int64_t qr0 = head0 + grp, qr1 = head0 + grp + 8;
        if (pre) {
            qr0 = s_qrow[grp];
            qr1 = G16 ? s_qrow[grp + 8] : -1;
            r0 = qr0 >= 0;
            r1 = qr1 >= 0;
        }
        const __nv_bfloat16* q0 = q + (r0 ? qr0 : 0) * D;
        const __nv_bfloat16* q1 = q + (r1 ? qr1 : 0) * D;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            const int d0 = ks * 16 + 2 * tig;
            qa[ks][0] = r0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
            qa[ks][1] = r1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
            qa[ks][2] = r0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
            qa[ks][3] = r1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
        }
    }

    // tokens of the row this CTA walks (a member: past its shared blocks)
    const int32_t T = pre ? T_raw : max(0, clamp_len(a, T_raw) - skip);
    const int32_t nparts = (int32_t)(((int64_t)T + P - 1) / P);
    if (T == 0) {
        if (p == 0 && direct)
            for (int32_t x = tid; x < G * D; x += C::kThreads)
                out[head0 * D + x] = __float2bfloat16_rn(0.f);
        return;
    }
    if (p >= nparts) return;

    int32_t n = min(P, T - t0);
    // a prefix CTA loads the keys up to its longest member's last one; each
    // row masks the keys past its own member's length (rlim0 / rlim1)
    int32_t rlim0 = n, rlim1 = n;
    if (pre) {
        int32_t most = 0;
#pragma unroll
        for (int r = 0; r < C::kRows; ++r) most = max(most, s_lim[r]);
        n = min(n, most);
        rlim0 = s_lim[grp];
        rlim1 = G16 ? s_lim[grp + 8] : 0;
    }
    const int32_t nblk = (n + BS - 1) / BS;
    const int32_t nchunk = (n + C::kChunk - 1) / C::kChunk;
    // Fused append: the CTA whose partition holds position T - 1 takes that
    // token's K and V rows from k_new / v_new.  Lane l of the warp that owns
    // its chunk holds 16 bytes (lanes 0-15 K, 16-31 V, eight columns each),
    // loaded here so the load overlaps the first tile copies; they replace
    // row rnew of the chunk's tile once its copy has landed.  A clamped
    // (reported) length appends nothing.
    int32_t cnew = -1, rnew = 0;
    uint4 nrow = make_uint4(0u, 0u, 0u, 0u);
    const bool npiece = (lane & 15) * 8 < D;
    if (!CAS && a.k_new != nullptr && T == T_raw && T - 1 >= t0 && T - 1 < t0 + n) {
        cnew = (T - 1 - t0) / C::kChunk;
        rnew = T - 1 - t0 - cnew * C::kChunk;
        if (cnew % C::kWarps == warp && npiece) {
            const __nv_bfloat16* src =
                static_cast<const __nv_bfloat16*>(lane < 16 ? a.k_new : a.v_new);
            nrow = *reinterpret_cast<const uint4*>(src + ((int64_t)i * a.num_kv_heads + g) * D +
                                                   (lane & 15) * 8);
        }
    }
#pragma unroll
    for (int r = 0; r < kIdsPerThread; ++r) {
        const int32_t b = tid + r * C::kThreads;
        if (b < nblk) {
            int32_t id = raw_ids[r];
            if (id < 0 || id >= a.num_blocks) {
                raise_error(PA_DEVERR_TABLE_ENTRY);
                id = -1;
            }
            ids[b] = id;
        }
    }
    __syncthreads();

    // warp w takes chunks w, w + 4, w + 8, ... of the partition
    const int32_t my_count = nchunk > warp ? (nchunk - warp + C::kWarps - 1) / C::kWarps : 0;
    const uint32_t ring_u = smem_u32(sm) + warp * C::kStages * C::kStageBytes;
    const uint32_t bar0 = smem_u32(&bars[warp * C::kStages]);
    const int32_t hkv = a.num_kv_heads;
    const uint64_t policy = l2_policy_evict_first();

    // A chunk is usable when its block(s) passed the table check; a chunk
    // touching a bad entry is skipped whole (its output is undefined anyway,
    // and the error bit is set).
    auto chunk_ok = [&](int32_t c) -> bool {
        if (BS >= C::kChunk) return ids[c / cpb] >= 0;
        return ids[2 * c] >= 0 && (2 * c + 1 >= nblk || ids[2 * c + 1] >= 0);
    };
    auto issue = [&](int32_t k) {   // lane 0 only
        const int32_t c = warp + k * C::kWarps;
        const int32_t st = k % C::kStages;
        const uint32_t bar = bar0 + 8 * st;
        if (!chunk_ok(c)) {
            mbar_arrive(bar);
            return;
        }
        const uint32_t dst = ring_u + st * C::kStageBytes;
        fence_proxy_async_smem();
        if (BS >= C::kChunk) {
            const int32_t blk = c / cpb;
            const int32_t y = (c - blk * cpb) * C::kChunk;
            const int32_t z = ids[blk] * hkv + g;
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
            // B = 8: rows 0-7 from block 2c, rows 8-15 from block 2c+1 (if any)
            const int32_t halves = 2 * c + 1 < nblk ? 2 : 1;
            mbar_arrive_expect_tx(bar, halves * (C::kStageBytes / 2));
            for (int h = 0; h < halves; ++h) {
                const int32_t z = ids[2 * c + h] * hkv + g;
#pragma unroll
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d_hint(dst + b * C::kBoxBytes + h * 1024, &tmap_k,
                                     b * C::kBoxCols, 0, z, bar, policy);
#pragma unroll
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d_hint(dst + C::kTileBytes + b * C::kBoxBytes + h * 1024, &tmap_v,
                                     b * C::kBoxCols, 0, z, bar, policy);
            }
        }
    };
    if (lane == 0) {
        const int32_t pre = my_count < C::kStages ? my_count : C::kStages;
        for (int32_t k = 0; k < pre; ++k) issue(k);
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[C::kDTiles][4];
#pragma unroll
    for (int nd = 0; nd < C::kDTiles; ++nd) acc[nd][0] = acc[nd][1] = acc[nd][2] = acc[nd][3] = 0.f;

    const int32_t lm = lane >> 3, lr = lane & 7;   // ldmatrix: matrix index, row in matrix
    int32_t k = 0;
    bool failed = false;
    for (; k < my_count; ++k) {
        const int32_t st = k % C::kStages;
        const bool ok = mbar_wait_bounded(bar0 + 8 * st, (k / C::kStages) & 1, kWaitLimitCycles);
        if (__any_sync(0xffffffffu, !ok)) {
            failed = true;
            break;
        }
        const int32_t c = warp + k * C::kWarps;
        if (chunk_ok(c)) {
            const uint32_t kb = ring_u + st * C::kStageBytes;
            const uint32_t vb = kb + C::kTileBytes;
            const int32_t nvalid = min(C::kChunk, n - c * C::kChunk);
            if (nvalid < C::kChunk) {
                // Unused rows of a sequence's last block may hold anything
                // (even NaN); their weights are 0, so clear their V rows.
                uint8_t* vt = sm + warp * C::kStages * C::kStageBytes + st * C::kStageBytes +
                              C::kTileBytes;
                const int32_t chunks = (C::kChunk - nvalid) * 8;   // 16-byte pieces per box
                for (int32_t x = lane; x < C::kBoxes * chunks; x += 32) {
                    const int32_t b = x / chunks, r = x - b * chunks;
                    *reinterpret_cast<uint4*>(vt + b * C::kBoxBytes + nvalid * 128 + r * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            if (!CAS && c == cnew) {
                // the appended token: its rows replace row rnew of the K and
                // V tiles (same 128-byte swizzle as the copy), and sub-group 0
                // stores them to the caches for later calls
                if (npiece) {
                    const int32_t pc = lane & 15;
                    uint8_t* tile = sm + warp * C::kStages * C::kStageBytes + st * C::kStageBytes +
                                    (lane < 16 ? 0 : C::kTileBytes);
                    *reinterpret_cast<uint4*>(tile + (pc >> 3) * C::kBoxBytes + rnew * 128 +
                                              (((pc & 7) ^ (rnew & 7)) << 4)) = nrow;
                    if (sg == 0) {
                        const int32_t off = T - 1 - t0, pos = T - 1 - (T - 1) / BS * BS;
                        const int64_t crow = ((int64_t)ids[off / BS] * hkv + g) * BS + pos;
                        void* cache = const_cast<void*>(lane < 16 ? a.k_cache : a.v_cache);
                        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(cache) +
                                                  crow * D + pc * 8) = nrow;
                    }
                }
                __syncwarp();
            }

            // S = Q . K^T for the 16 tokens of the chunk (two n-tiles of 8)
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
            // scale, mask, row max
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    // CAS: per row (a prefix CTA's rows end at their members'
                    // lengths); otherwise one end for all rows
                    const int32_t col = c * C::kChunk + nt * 8 + 2 * tig + e;
                    const bool valid = CAS ? col < rlim0 : nt * 8 + 2 * tig + e < nvalid;
                    const bool valid1 = CAS ? col < rlim1 : valid;
                    s[nt][e] = valid ? s[nt][e] * a.scale_log2 : -INFINITY;
                    mx0 = fmaxf(mx0, s[nt][e]);
                    if (G16) {
                        s[nt][2 + e] = valid1 ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
                        mx1 = fmaxf(mx1, s[nt][2 + e]);
                    }
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            const float mn0 = fmaxf(m0, mx0);
            // CAS: a prefix row may have seen no key yet (m stays -inf, its
            // weights are 0); the reference then is 0, not -inf - -inf
            const float ref0 = CAS && mn0 == -INFINITY ? 0.f : mn0;
            const float al0 = exp2f(m0 - ref0);
            m0 = mn0;
            float al1 = 1.f, ref1 = 0.f;
            if (G16) {
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn1 = fmaxf(m1, mx1);
                ref1 = CAS && mn1 == -INFINITY ? 0.f : mn1;
                al1 = exp2f(m1 - ref1);
                m1 = mn1;
            }
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
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
            for (int nd = 0; nd < C::kDTiles; ++nd) {
                acc[nd][0] *= al0;
                acc[nd][1] *= al0;
                acc[nd][2] *= G16 ? al1 : al0;     // G <= 8: the lo products of rows 0-7
                acc[nd][3] *= G16 ? al1 : al0;
            }
            // acc += P . V (P reused from the S registers as the A operand).
            // P = hi + lo, both bf16: hi is P rounded, lo the rounding error
            // rounded again, so P V keeps about 16 significant bits of each
            // weight instead of 8.  With G <= 8 the MMA's rows 8-15 are free
            // and carry the lo parts of rows 0-7 (their products land in this
            // thread's accumulators 2-3 and are added to 0-1 at the end); with
            // G > 8 the lo parts take a second product (cheap: this kernel
            // waits on HBM, not on the tensor pipe).
            uint32_t pf[4], pl[4];
            auto split = [](float x, float y, uint32_t& hi, uint32_t& lo) {
                hi = pack_bf16x2(x, y);
                lo = pack_bf16x2(x - __uint_as_float(hi << 16),
                                 y - __uint_as_float(hi & 0xffff0000u));
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
                    if (G16) {
                        mma_bf16_16816(acc[2 * dp], pl, b0, b1);
                        mma_bf16_16816(acc[2 * dp + 1], pl, b2, b3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && k + C::kStages < my_count) issue(k + C::kStages);
    }

    griddep_launch_dependents();   // the merge kernel may be scheduled now
    if (failed) {
        // drain this warp's copies still in flight (bounded), then report
        const int32_t last = min(my_count, k + C::kStages);
        for (int32_t kk = k; kk < last; ++kk)
            mbar_wait_bounded(bar0 + 8 * (kk % C::kStages), (kk / C::kStages) & 1,
                              kWaitLimitCycles);
        if (lane == 0) {
            raise_error(PA_DEVERR_TIMEOUT);
            atomicOr(&s_fail, 1);
        }
    }

    if (!G16) {
#pragma unroll
        for (int nd = 0; nd < C::kDTiles; ++nd) {
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
    __syncthreads();   // every warp is done with its ring

    float* cm = reinterpret_cast<float*>(sm);      // [kWarps][kRows]
    float* cl = cm + C::kWarps * C::kRows;          // [kWarps][kRows]
    float* ca = cl + C::kWarps * C::kRows;          // [kWarps][kRows][D]
    const bool fail = s_fail != 0;
    if (!fail) {
        if (tig == 0) {
            cm[warp * C::kRows + grp] = m0;
            cl[warp * C::kRows + grp] = l0;
            if (G16) {
                cm[warp * C::kRows + grp + 8] = m1;
                cl[warp * C::kRows + grp + 8] = l1;
            }
        }
#pragma unroll
        for (int nd = 0; nd < C::kDTiles; ++nd) {
            const int d = nd * 8 + 2 * tig;
            float* r0 = ca + (warp * C::kRows + grp) * D + d;
            r0[0] = acc[nd][0];
            r0[1] = acc[nd][1];
            if (G16) {
                float* r1 = ca + (warp * C::kRows + grp + 8) * D + d;
                r1[0] = acc[nd][2];
                r1[1] = acc[nd][3];
            }
        }
    }
    __syncthreads();

    for (int32_t x = tid; x < G * D; x += C::kThreads) {
        const int32_t h = x / D, d = x - h * D;
        float M = -INFINITY, L = 0.f, A = 0.f;
        if (!fail) {
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, cm[w * C::kRows + h]);
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) {
                const float mw = cm[w * C::kRows + h];
                if (mw != -INFINITY) {
                    const float e = exp2f(mw - M);
                    L += e * cl[w * C::kRows + h];
                    A += e * ca[(w * C::kRows + h) * D + d];
                }
            }
        }
        if (nparts == 1 && direct) {
            out[(head0 + h) * D + d] = __float2bfloat16_rn(L > 0.f ? A / L : 0.f);
        } else {
            // a prefix CTA's partials go to slot p of its rows' cells; a
            // member's after its group's prefix slots
            const int64_t qr = pre ? s_qrow[h] : head0 + h;
            if (qr >= 0) {
                const int64_t cell = qr * a.max_parts + slot0 + p;
                a.ws_acc[cell * D + d] = A;
                if (d == 0) {
                    a.ws_ml[2 * cell] = M;
                    a.ws_ml[2 * cell + 1] = L;
                }
            }
        }
    }
}

}  // namespace pa
