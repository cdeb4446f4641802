// prefill_tiled.cuh -- multi-query (chunked prefill) paged attention on CUDA
// cores for the shapes the tcgen05 kernel does not take: fp32 caches, head
// dims other than 64 and 128 (up to 256, rows of whole 16-byte pieces),
// block sizes other than 8 or a multiple of 16, negative scales.  Same
// definition as the other prefill kernels: sequence i's packed query rows are
// its last L_i positions, and the row at position p attends to keys 0..p
// ("vLLM source walkthrough: PagedAttention and Continuous Batching" §2.8;
// "Efficient Memory Management for LLM Serving with PagedAttention" paper
// notes, blockwise attention example: one softmax over all visible keys,
// accumulated block by block).
//
// One CTA of 128 threads per (query tile, kv head x sub-group, sequence).  A
// tile is R = 16 RPT rows, a row being a (token, query head) pair with the
// head fastest, so the heads of a token share every K/V byte the CTA reads.
// Keys are walked in chunks of KC through a double buffer in shared memory,
// filled with 16-byte cp.async copies through the block table (the wait is
// the copy engine's own group wait: nothing spins).  Thread (rg, kg), rg =
// tid / 8 and kg = tid % 8, owns rows rg RPT .. rg RPT + RPT - 1:
//   - scores of keys kg, kg + 8, ... of the chunk (K rows padded by 16 bytes,
//     so the eight threads of a row group read eight different banks);
//   - the row's online softmax, shared by the eight threads of its group
//     through shuffles (running max m, sum l, rescale a, base 2: q is scaled
//     by scale log2(e) when it is staged);
//   - P goes through shared memory to the same eight threads, which own
//     float4 column groups kg, kg + 8, ... of the row's accumulator:
//     acc = a acc + sum_k p[k] V[k][:].
#pragma once

#include "cp_async.cuh"
#include "prefill_args.cuh"

namespace pa {

constexpr int kPtThreads = 128;

// Row and column split for a head dim: RPT rows a thread (tile of 16 RPT
// rows), NF float4 column groups a thread, KC keys a chunk.
template <int RPT, int NF, int KC>
struct PrefillTiledCfg {
    static constexpr int kRows = 16 * RPT;
    static constexpr int kKeysPerThread = KC / 8;
    static_assert(KC % 8 == 0 && NF >= 1 && RPT >= 1, "tile shape");
    // dynamic shared bytes: q [rows][D] fp32 | K, V double buffer [KC][row + 16] | P [rows][KC]
    static size_t smem_bytes(int32_t head_dim, int32_t elem) {
        const size_t stride = (size_t)head_dim * elem + 16;
        return (size_t)kRows * head_dim * 4 + 2 * 2 * (size_t)KC * stride + (size_t)kRows * KC * 4;
    }
};

// Four consecutive values of a shared-memory row as floats (8- or 16-byte
// aligned).
template <typename E>
__device__ __forceinline__ float4 smem_load4(const uint8_t* p) {
    if constexpr (sizeof(E) == 2) {
        const uint2 x = *reinterpret_cast<const uint2*>(p);
        return make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xffff0000u),
                           __uint_as_float(x.y << 16), __uint_as_float(x.y & 0xffff0000u));
    } else {
        return *reinterpret_cast<const float4*>(p);
    }
}

template <typename E, int RPT, int NF, int KC>
__global__ void __launch_bounds__(kPtThreads)
prefill_tiled_kernel(const PrefillArgs a) {
    using C = PrefillTiledCfg<RPT, NF, KC>;
    constexpr int R = C::kRows, KPT = C::kKeysPerThread;
    constexpr int kE = (int)sizeof(E);
    extern __shared__ __align__(16) uint8_t sm_pt[];
    griddep_wait();                 // inputs may come from the previous kernel
    const int32_t tid = threadIdx.x, rg = tid >> 3, kg = tid & 7;
    const int32_t D = a.head_dim, G = a.group, BS = a.block_size;
    // a tile: QT tokens x HT heads (the last R mod HT rows idle); groups of
    // more than R heads take several CTAs (sub-groups) per kv head
    const int32_t HT = min(G, R), QT = R / HT;
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
    const int32_t rowb = D * kE, stride = rowb + 16, ppr = rowb / 16;
    float* qs = reinterpret_cast<float*>(sm_pt);                          // [R][D]
    uint8_t* kvs = sm_pt + (size_t)R * D * 4;                             // [2][K, V][KC][stride]
    float* ps = reinterpret_cast<float*>(kvs + 2 * 2 * KC * stride);      // [R][KC]

    const E* q = static_cast<const E*>(a.q);
    const int64_t head_base = (int64_t)g * G + sg * HT;
    for (int32_t x = tid; x < R * D; x += kPtThreads) {
        const int32_t rho = x / D, d = x - rho * D;
        const int32_t tk = rho / HT, hh = rho - tk * HT;
        float v = 0.f;
        if (tk < nt && hh < hs) {
            const int64_t row = (int64_t)(q0 + j0 + tk) * a.num_q_heads + head_base + hh;
            v = Elem<E>::to_float(q[row * D + d]) * a.scale_log2;
        }
        qs[x] = v;
    }

    // Copies of chunk c (keys c KC ..) into buffer c & 1: 16-byte pieces
    // through the block table; keys past the tile's last position and keys
    // behind a bad table entry are filled with zeros.
    const E* kc = static_cast<const E*>(a.k_cache);
    const E* vc = static_cast<const E*>(a.v_cache);
    const int32_t* table = a.block_tables + (int64_t)i * a.max_blocks;
    auto issue = [&](int32_t c) {
        uint8_t* kb = kvs + (c & 1) * 2 * KC * stride;
        uint8_t* vb = kb + KC * stride;
        for (int32_t x = tid; x < KC * ppr; x += kPtThreads) {
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
            cp_async16(smem_u32(kb + k * stride + piece * 16),
                       reinterpret_cast<const uint8_t*>(kc + off) + piece * 16, bytes);
            cp_async16(smem_u32(vb + k * stride + piece * 16),
                       reinterpret_cast<const uint8_t*>(vc + off) + piece * 16, bytes);
        }
    };

    // this thread's rows: validity and positions
    bool rvalid[RPT];
    int32_t rpos[RPT];
#pragma unroll
    for (int32_t r = 0; r < RPT; ++r) {
        const int32_t rho = rg * RPT + r, tk = rho / HT, hh = rho - tk * HT;
        rvalid[r] = tk < nt && hh < hs;
        rpos[r] = pbase + tk;
    }
    float m[RPT], l[RPT];
    float4 acc[RPT][NF];
#pragma unroll
    for (int32_t r = 0; r < RPT; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int32_t f = 0; f < NF; ++f) acc[r][f] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    issue(0);
    cp_async_commit();
    for (int32_t c = 0; c < nch; ++c) {
        if (c + 1 < nch) {         // next chunk in flight while this one is used
            issue(c + 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();           // chunk c (and, at c = 0, q) visible to every thread
        const uint8_t* kb = kvs + (c & 1) * 2 * KC * stride;
        const uint8_t* vb = kb + KC * stride;

        // scores of rows rg RPT + r and keys kg + 8 j
        float s[RPT][KPT];
#pragma unroll
        for (int32_t r = 0; r < RPT; ++r)
#pragma unroll
            for (int32_t j = 0; j < KPT; ++j) s[r][j] = 0.f;
#pragma unroll 4
        for (int32_t d4 = 0; d4 < D / 4; ++d4) {
            float4 qv[RPT], kv4[KPT];
#pragma unroll
            for (int32_t r = 0; r < RPT; ++r)
                qv[r] = *reinterpret_cast<const float4*>(qs + (rg * RPT + r) * D + 4 * d4);
#pragma unroll
            for (int32_t j = 0; j < KPT; ++j)
                kv4[j] = smem_load4<E>(kb + (kg + 8 * j) * stride + d4 * 4 * kE);
#pragma unroll
            for (int32_t r = 0; r < RPT; ++r)
#pragma unroll
                for (int32_t j = 0; j < KPT; ++j) {
                    float x = s[r][j];
                    x = fmaf(qv[r].x, kv4[j].x, x);
                    x = fmaf(qv[r].y, kv4[j].y, x);
                    x = fmaf(qv[r].z, kv4[j].z, x);
                    x = fmaf(qv[r].w, kv4[j].w, x);
                    s[r][j] = x;
                }
        }

        // causal mask, online softmax per row (its eight threads), p to
        // shared memory for the eight threads' P V
        const int32_t t0 = c * KC;
        float al[RPT];
#pragma unroll
        for (int32_t r = 0; r < RPT; ++r) {
            float mx = -INFINITY;
#pragma unroll
            for (int32_t j = 0; j < KPT; ++j) {
                const int32_t t = t0 + kg + 8 * j;
                s[r][j] = rvalid[r] && t <= rpos[r] ? s[r][j] : -INFINITY;
                mx = fmaxf(mx, s[r][j]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            const float mn = fmaxf(m[r], mx);
            const float mref = mn == -INFINITY ? 0.f : mn;    // no visible key yet
            al[r] = exp2f(m[r] - mref);                        // 0 while m = -inf
            float sum = 0.f;
#pragma unroll
            for (int32_t j = 0; j < KPT; ++j) {
                s[r][j] = exp2f(s[r][j] - mref);               // 0 for masked keys
                sum += s[r][j];
                ps[(rg * RPT + r) * KC + kg + 8 * j] = s[r][j];
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            l[r] = l[r] * al[r] + sum;
            m[r] = mn;
        }
        __syncwarp();              // a row group's p, written by its own warp

#pragma unroll
        for (int32_t r = 0; r < RPT; ++r)
#pragma unroll
            for (int32_t f = 0; f < NF; ++f) {
                acc[r][f].x *= al[r];
                acc[r][f].y *= al[r];
                acc[r][f].z *= al[r];
                acc[r][f].w *= al[r];
            }
#pragma unroll 2
        for (int32_t k4 = 0; k4 < KC; k4 += 4) {
            float4 pv[RPT];
#pragma unroll
            for (int32_t r = 0; r < RPT; ++r)
                pv[r] = *reinterpret_cast<const float4*>(ps + (rg * RPT + r) * KC + k4);
#pragma unroll
            for (int32_t kk = 0; kk < 4; ++kk) {
                const uint8_t* vrow = vb + (k4 + kk) * stride;
#pragma unroll
                for (int32_t f = 0; f < NF; ++f) {
                    const int32_t col = 4 * (kg + 8 * f);
                    if (col < D) {
                        const float4 v = smem_load4<E>(vrow + col * kE);
#pragma unroll
                        for (int32_t r = 0; r < RPT; ++r) {
                            const float p = kk == 0 ? pv[r].x : kk == 1 ? pv[r].y
                                          : kk == 2 ? pv[r].z : pv[r].w;
                            acc[r][f].x = fmaf(p, v.x, acc[r][f].x);
                            acc[r][f].y = fmaf(p, v.y, acc[r][f].y);
                            acc[r][f].z = fmaf(p, v.z, acc[r][f].z);
                            acc[r][f].w = fmaf(p, v.w, acc[r][f].w);
                        }
                    }
                }
            }
        }
        __syncthreads();           // buffer c & 1 and p are free
    }
    griddep_launch_dependents();

    E* out = static_cast<E*>(a.out);
#pragma unroll
    for (int32_t r = 0; r < RPT; ++r) {
        if (!rvalid[r]) continue;
        const int32_t rho = rg * RPT + r, tk = rho / HT, hh = rho - tk * HT;
        const int64_t row = (int64_t)(q0 + j0 + tk) * a.num_q_heads + head_base + hh;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
#pragma unroll
        for (int32_t f = 0; f < NF; ++f) {
            const int32_t col = 4 * (kg + 8 * f);
            if (col >= D) continue;
            const float4 o = acc[r][f];
            if constexpr (kE == 2) {
                uint2 w;
                w.x = pack_bf16x2(o.x * inv, o.y * inv);
                w.y = pack_bf16x2(o.z * inv, o.w * inv);
                *reinterpret_cast<uint2*>(out + row * D + col) = w;
            } else {
                *reinterpret_cast<float4*>(out + row * D + col) =
                    make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            }
        }
    }
}

}  // namespace pa
