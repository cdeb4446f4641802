// prefill_mma.cuh -- bf16 multi-query (chunked prefill) paged attention on
// the warp-level tensor-core path (mma.sync m16n8k16) for the shapes the
// tcgen05 kernel does not take: head dims other than 64 and 128 (multiples of
// 16 up to 256), block sizes other than 8 or a multiple of 16, negative
// scales.  Same definition as the other prefill kernels ("vLLM source
// walkthrough: PagedAttention and Continuous Batching" §2.8: the row at
// position p attends to keys 0..p of its sequence through the block table;
// "Efficient Memory Management for LLM Serving with PagedAttention" paper
// notes, blockwise attention example: one softmax over all visible keys,
// accumulated block by block).
//
// One CTA of four warps per (64-row query tile, kv head x sub-group,
// sequence); a row is a (token, query head) pair with the head fastest, so
// the heads of a token share every K/V byte.  Q is staged in shared memory;
// keys arrive in chunks of KC through a double buffer of 16-byte cp.async
// copies through the block table, every row padded by 16 bytes so that the
// eight rows an ldmatrix reads sit in eight different bank groups.  Warp w
// owns rows 16 w .. 16 w + 15:
//   S = Q K^T               (ldmatrix of Q and K, fp32 accumulators)
//   online softmax in base 2 on the S fragments (scale log2 e applied to S)
//   O += P V                (P from the S registers as bf16 hi + lo, V by
//                            ldmatrix.trans)
#pragma once

#include "prefill_tiled.cuh"

namespace pa {

constexpr int kPmThreads = 128;
constexpr int kPmRows = 64;   // 16 rows a warp

// DMAX: largest head dim of the instance (128 or 256); KC: keys a chunk.
template <int DMAX, int KC>
struct PrefillMmaCfg {
    static_assert(DMAX % 16 == 0 && KC % 16 == 0, "tile shape");
    // dynamic shared bytes: q [64][row + 16] | K, V double buffer [KC][row + 16]
    static size_t smem_bytes(int32_t head_dim) {
        const size_t stride = (size_t)head_dim * 2 + 16;
        return kPmRows * stride + 2 * 2 * (size_t)KC * stride;
    }
};

template <int DMAX, int KC>
__global__ void __launch_bounds__(kPmThreads)
prefill_mma_kernel(const PrefillArgs a) {
    constexpr int NT = KC / 8;           // key n-tiles of S
    constexpr int DT = DMAX / 8;         // column n-tiles of O
    extern __shared__ __align__(16) uint8_t sm_pm[];
    griddep_wait();                      // inputs may come from the previous kernel
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t grp = lane >> 2, tig = lane & 3;
    const int32_t lm = lane >> 3, lr = lane & 7;      // ldmatrix: matrix, row in matrix
    const int32_t D = a.head_dim, G = a.group, BS = a.block_size;
    const int32_t HT = min(G, kPmRows), QT = kPmRows / HT;
    const int32_t nsub = (G + HT - 1) / HT;
    const int32_t g = blockIdx.y / nsub, sg = blockIdx.y - g * nsub;
    const int32_t i = blockIdx.z;
    const int32_t q0 = a.query_start[i], L = a.query_start[i + 1] - q0;
    const int32_t T = clamp_len(a, a.seq_lens[i]);
    if (L > T) {
        if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int32_t j0 = blockIdx.x * QT;
    if (j0 >= L) return;
    const int32_t nt = min(QT, L - j0);                // tokens of this tile
    const int32_t hs = min(HT, G - sg * HT);           // heads of this tile
    const int32_t pbase = T - L + j0;                  // position of the tile's first token
    const int32_t nkeys = pbase + nt;                  // keys 0 .. pbase + nt - 1
    const int32_t nch = (nkeys + KC - 1) / KC;
    const int32_t rowb = D * 2, stride = rowb + 16, ppr = rowb / 16;
    uint8_t* qsm = sm_pm;                                       // [64][stride]
    uint8_t* kvs = sm_pm + kPmRows * stride;                    // [2][K, V][KC][stride]
    const uint32_t q_u = smem_u32(qsm), kv_u = smem_u32(kvs);

    // Q rows of the tile (zeros for idle rows)
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    const int64_t head_base = (int64_t)g * G + sg * HT;
    for (int32_t x = tid; x < kPmRows * ppr; x += kPmThreads) {
        const int32_t rho = x / ppr, piece = x - rho * ppr;
        const int32_t tk = rho / HT, hh = rho - tk * HT;
        const bool ok = tk < nt && hh < hs;
        const int64_t row = ok ? (int64_t)(q0 + j0 + tk) * a.num_q_heads + head_base + hh : 0;
        cp_async16(q_u + rho * stride + piece * 16,
                   reinterpret_cast<const uint8_t*>(q + row * D) + piece * 16, ok ? 16u : 0u);
    }

    const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
    const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;
    auto issue = [&](int32_t c) {
        const uint32_t kb = kv_u + (c & 1) * 2 * KC * stride;
        const uint32_t vb = kb + KC * stride;
        for (int32_t x = tid; x < KC * ppr; x += kPmThreads) {
            const int32_t k = x / ppr, piece = x - k * ppr;
            const int32_t t = c * KC + k;
            int32_t id = -1;
            if (t < nkeys) {
                id = table[t / BS];
                if (id < 0 || id >= a.num_blocks) {
                    raise_error(PA_DEVERR_TABLE_ENTRY);
                    id = -1;
                }
            }
            const int64_t off = id >= 0 ? (((int64_t)id * a.num_kv_heads + g) * BS + t % BS) * D : 0;
            const uint32_t bytes = id >= 0 ? 16u : 0u;
            cp_async16(kb + k * stride + piece * 16,
                       reinterpret_cast<const uint8_t*>(kc + off) + piece * 16, bytes);
            cp_async16(vb + k * stride + piece * 16,
                       reinterpret_cast<const uint8_t*>(vc + off) + piece * 16, bytes);
        }
    };

    // this lane's two rows: warp * 16 + grp (half 0) and + 8 (half 1)
    bool rvalid[2];
    int32_t rpos[2];
#pragma unroll
    for (int32_t h = 0; h < 2; ++h) {
        const int32_t rho = warp * 16 + grp + 8 * h, tk = rho / HT, hh = rho - tk * HT;
        rvalid[h] = tk < nt && hh < hs;
        rpos[h] = pbase + tk;
    }
    // the warp's last position: chunks past it are fully masked for the warp
    int32_t wpos = -1;
    {
        const int32_t rho = warp * 16 + 15;
        const int32_t tk = min(rho / HT, nt - 1);
        if (warp * 16 / HT < nt) wpos = pbase + tk;
    }
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float acc[DT][4];
#pragma unroll
    for (int32_t nd = 0; nd < DT; ++nd) acc[nd][0] = acc[nd][1] = acc[nd][2] = acc[nd][3] = 0.f;

    issue(0);
    cp_async_commit();             // q and chunk 0
    for (int32_t c = 0; c < nch; ++c) {
        if (c + 1 < nch) {         // next chunk in flight while this one is used
            issue(c + 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();           // chunk c (and q) visible to every warp
        const int32_t t0 = c * KC;
        if (t0 <= wpos) {          // some key of the chunk is visible to the warp's rows
            const uint32_t kb = kv_u + (c & 1) * 2 * KC * stride;
            const uint32_t vb = kb + KC * stride;

            // S = Q K^T: per 16 columns of D, one Q fragment against every
            // 16-key pair of n-tiles
            float s[NT][4];
#pragma unroll
            for (int32_t n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
            for (int32_t ks = 0; ks < DMAX / 16; ++ks) {
                if (ks < D / 16) {
                    uint32_t qa[4];
                    ldsm_x4(q_u + (warp * 16 + (lm & 1) * 8 + lr) * stride + (ks * 16 + (lm >> 1) * 8) * 2,
                            qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
                    for (int32_t kp = 0; kp < KC / 16; ++kp) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kb + (kp * 16 + (lm >> 1) * 8 + lr) * stride +
                                    (ks * 16 + (lm & 1) * 8) * 2,
                                b0, b1, b2, b3);
                        mma_bf16_16816(s[2 * kp], qa, b0, b1);
                        mma_bf16_16816(s[2 * kp + 1], qa, b2, b3);
                    }
                }
            }

            // scale, causal mask, online softmax of rows grp (h = 0) and
            // grp + 8 (h = 1); a row's columns are spread over its 4 lanes
            float al[2];
#pragma unroll
            for (int32_t h = 0; h < 2; ++h) {
                float mx = -INFINITY;
#pragma unroll
                for (int32_t n = 0; n < NT; ++n)
#pragma unroll
                    for (int32_t e = 0; e < 2; ++e) {
                        const int32_t t = t0 + n * 8 + 2 * tig + e;
                        float& x = s[n][2 * h + e];
                        x = rvalid[h] && t <= rpos[h] ? x * a.scale_log2 : -INFINITY;
                        mx = fmaxf(mx, x);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(m[h], mx);
                const float mref = mn == -INFINITY ? 0.f : mn;   // no visible key yet
                al[h] = exp2f(m[h] - mref);                       // 0 while m = -inf
                float sum = 0.f;
#pragma unroll
                for (int32_t n = 0; n < NT; ++n)
#pragma unroll
                    for (int32_t e = 0; e < 2; ++e) {
                        float& x = s[n][2 * h + e];
                        x = exp2f(x - mref);                      // 0 for masked keys
                        sum += x;
                    }
                l[h] = l[h] * al[h] + sum;                        // this lane's columns only
                m[h] = mn;
            }
#pragma unroll
            for (int32_t nd = 0; nd < DT; ++nd) {
                acc[nd][0] *= al[0];
                acc[nd][1] *= al[0];
                acc[nd][2] *= al[1];
                acc[nd][3] *= al[1];
            }

            // O += P V, P from the S registers (two key n-tiles = one k step).
            // P = hi + lo, both bf16 (the rounding error of hi rounded again):
            // two products against the same V fragments keep about 16
            // significant bits of each weight instead of 8.
#pragma unroll
            for (int32_t kp = 0; kp < KC / 16; ++kp) {
                uint32_t pf[4], pl[4];
                split_bf16x2(s[2 * kp][0], s[2 * kp][1], pf[0], pl[0]);
                split_bf16x2(s[2 * kp][2], s[2 * kp][3], pf[1], pl[1]);
                split_bf16x2(s[2 * kp + 1][0], s[2 * kp + 1][1], pf[2], pl[2]);
                split_bf16x2(s[2 * kp + 1][2], s[2 * kp + 1][3], pf[3], pl[3]);
#pragma unroll
                for (int32_t dp = 0; dp < DMAX / 16; ++dp) {
                    if (dp < D / 16) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(vb + (kp * 16 + (lm & 1) * 8 + lr) * stride +
                                          (dp * 16 + (lm >> 1) * 8) * 2,
                                      b0, b1, b2, b3);
                        mma_bf16_16816(acc[2 * dp], pf, b0, b1);
                        mma_bf16_16816(acc[2 * dp + 1], pf, b2, b3);
                        mma_bf16_16816(acc[2 * dp], pl, b0, b1);
                        mma_bf16_16816(acc[2 * dp + 1], pl, b2, b3);
                    }
                }
            }
        }
        __syncthreads();           // buffer c & 1 is free
    }
    griddep_launch_dependents();

    // row sums over the row's 4 lanes, then out = O / l
#pragma unroll
    for (int32_t h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
    for (int32_t h = 0; h < 2; ++h) {
        if (!rvalid[h]) continue;
        const int32_t rho = warp * 16 + grp + 8 * h, tk = rho / HT, hh = rho - tk * HT;
        const int64_t row = (int64_t)(q0 + j0 + tk) * a.num_q_heads + head_base + hh;
        const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll
        for (int32_t nd = 0; nd < DT; ++nd) {
            if (nd < D / 8)
                *reinterpret_cast<uint32_t*>(out + row * D + nd * 8 + 2 * tig) =
                    pack_bf16x2(acc[nd][2 * h] * inv, acc[nd][2 * h + 1] * inv);
        }
    }
}

}  // namespace pa
