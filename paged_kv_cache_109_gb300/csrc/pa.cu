// pa.cu -- C-ABI entry points of libpa.so (declared in include/pa.h).
//
// Host side only: argument checks, kernel selection, split-K sizing, TMA
// descriptor encoding and launches on the caller's stream.  Every step of the
// computation runs in the kernels of the included headers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "debug_checks.h"
#include "decode_generic.cuh"
#include "decode_tiled.cuh"
#include "decode_config.cuh"
#include "decode_mma.cuh"
#include "decode_tma_mma.cuh"
#include "merge.cuh"
#include "prefill_generic.cuh"
#include "prefill_mma.cuh"
#include "prefill_tiled.cuh"
#include "prefill_ws.cuh"
#include "wait_check.cuh"
#include "write_kv.cuh"

namespace pa {
namespace {

bool desc_ok(const pa_cache_desc* c) {
    return c && c->num_blocks > 0 && c->block_size > 0 && c->num_kv_heads > 0 &&
           c->head_dim > 0 && (c->dtype == PA_F32 || c->dtype == PA_BF16);
}

int elem_bytes(const pa_cache_desc* c) { return c->dtype == PA_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- TMA descriptors -----------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Cache viewed as 3-D: (head_dim, block_size, num_blocks * Hkv); one box is a
// 64-column (128-byte) slice of 16 rows of one (block, head) tile, swizzled
// 128 B.
bool encode_cache_map(CUtensorMap* map, const void* base, const pa_cache_desc* c) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)c->head_dim, (cuuint64_t)c->block_size,
                          (cuuint64_t)c->num_blocks * (cuuint64_t)c->num_kv_heads};
    cuuint64_t strides[2] = {(cuuint64_t)c->head_dim * 2,
                             (cuuint64_t)c->head_dim * 2 * (cuuint64_t)c->block_size};
    cuuint32_t box[3] = {64, (cuuint32_t)std::min(16, c->block_size), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct MapCacheEntry {
    const void* base = nullptr;
    pa_cache_desc desc{};
    CUtensorMap map;
};

bool cached_map(CUtensorMap* out, const void* base, const pa_cache_desc* c, int slot) {
    thread_local MapCacheEntry entries[2];
    MapCacheEntry& e = entries[slot];
    if (e.base != base || std::memcmp(&e.desc, c, sizeof(*c)) != 0) {
        if (!encode_cache_map(&e.map, base, c)) {
            e.base = nullptr;
            return false;
        }
        e.base = base;
        e.desc = *c;
    }
    *out = e.map;
    return true;
}

// ---- launches ------------------------------------------------------------------

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream finishes; it waits for that kernel
// (griddepcontrol.wait) before reading any input.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PA_USE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename E, int W, int VEC>
cudaError_t launch_merge_k(dim3 grid, cudaStream_t st, const DecodeArgs& a) {
    return launch_pdl(merge_kernel<E, W, VEC>, grid, dim3(32 * W), 0, st, a);
}

// CTAs of merge_kernel<E, W, VEC> one SM holds (0 if unknown), per device.
template <typename E, int W, int VEC>
int merge_ctas_per_sm() {
    static int cached[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, merge_kernel<E, W, VEC>, 32 * W,
                                                          0) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

template <typename E, int VEC>
cudaError_t launch_merge_w(int warps, dim3 grid, cudaStream_t st, const DecodeArgs& a) {
    // fewer warps a pair while the grid would take more than one wave on
    // the GPU (a second wave of merge CTAs costs more than a warp's extra
    // chunk rounds); an unknown occupancy changes nothing
    const int64_t sms = std::max(1, device_sm_count());
    auto fits = [&](int w) {
        const int per = w == 8   ? merge_ctas_per_sm<E, 8, VEC>()
                        : w == 4 ? merge_ctas_per_sm<E, 4, VEC>()
                                 : merge_ctas_per_sm<E, 2, VEC>();
        return per <= 0 || (int64_t)grid.x <= per * sms;
    };
    while (warps > 1 && !fits(warps)) warps /= 2;
    switch (warps) {
        case 1: return launch_merge_k<E, 1, VEC>(grid, st, a);
        case 2: return launch_merge_k<E, 2, VEC>(grid, st, a);
        case 4: return launch_merge_k<E, 4, VEC>(grid, st, a);
        default: return launch_merge_k<E, 8, VEC>(grid, st, a);
    }
}

// The merge launch of a call: one CTA per (sequence, query head), after the
// partition kernel on the same stream (programmatic dependent launch); its
// warps are sized for typical_parts partitions (any count merges correctly).
template <typename E>
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t st, int32_t typical_parts) {
    const dim3 grid((unsigned)((int64_t)a.num_seqs * a.num_q_heads));
    const int warps = merge_warps(typical_parts);
    return a.head_dim % 4 == 0 ? launch_merge_w<E, 4>(warps, grid, st, a)
                               : launch_merge_w<E, 1>(warps, grid, st, a);
}


template <typename Kern>
bool set_smem(Kern kern, size_t bytes) {
    if (bytes <= 48 * 1024) return true;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)bytes) == cudaSuccess;
}

template <int D, bool G16, bool CAS>
cudaError_t launch_fast(dim3 grid, const CUtensorMap& mk, const CUtensorMap& mv,
                        const DecodeArgs& a, cudaStream_t st) {
    using C = TmaMmaCfg<D, G16>;
    auto kern = decode_tma_mma_kernel<D, G16, CAS>;
    if (!set_smem(kern, C::smem_bytes_max())) return cudaErrorInvalidValue;
    const size_t smem = C::smem_bytes(a.part_tokens, a.block_size);
    return launch_pdl(kern, grid, dim3(C::kThreads), smem, st, mk, mv, a);
}

template <typename E, int HB, int CH, int C>
cudaError_t launch_tiled_kernel(dim3 grid, size_t smem, cudaStream_t st, const DecodeArgs& a) {
    auto kern = decode_tiled_kernel<E, HB, CH, C>;
    if (!set_smem(kern, smem)) return cudaErrorInvalidValue;
    return launch_pdl(kern, grid, dim3(kTiledThreads), smem, st, a);
}

template <typename E, int CH, int C>
cudaError_t launch_tiled_hb(int32_t hb, dim3 grid, size_t smem, cudaStream_t st,
                            const DecodeArgs& a) {
    switch (hb) {
        case 1: return launch_tiled_kernel<E, 1, CH, C>(grid, smem, st, a);
        case 2: return launch_tiled_kernel<E, 2, CH, C>(grid, smem, st, a);
        case 4: return launch_tiled_kernel<E, 4, CH, C>(grid, smem, st, a);
        default: return launch_tiled_kernel<E, 8, CH, C>(grid, smem, st, a);
    }
}

// The tiled kernel's instance for the shape: heads per CTA rounded to a power
// of 2, chunk tokens and columns per lane from the row size (4 KB chunks:
// bf16 (16, 4) up to D = 128, else (8, 8); fp32 (16, 4) up to D = 64, (8, 4)
// up to 128, else (4, 8)).
cudaError_t dispatch_tiled(const pa_cache_desc* c, int32_t group, dim3 grid,
                           const DecodeArgs& a, cudaStream_t st) {
    const int32_t D = c->head_dim, e = elem_bytes(c);
    const int32_t hb = tiled_heads_rounded(tiled_sub_group(group));
    const size_t smem = tiled_smem_bytes(D, e, hb);
    const int32_t ch = tiled_chunk(D, e), cols = tiled_cols(D);
    if (c->dtype == PA_F32) {
        if (ch == 16 && cols == 4) return launch_tiled_hb<float, 16, 4>(hb, grid, smem, st, a);
        if (ch == 8 && cols == 4) return launch_tiled_hb<float, 8, 4>(hb, grid, smem, st, a);
        if (ch == 4 && cols == 8) return launch_tiled_hb<float, 4, 8>(hb, grid, smem, st, a);
    } else {
        if (ch == 16 && cols == 4)
            return launch_tiled_hb<__nv_bfloat16, 16, 4>(hb, grid, smem, st, a);
        if (ch == 8 && cols == 8)
            return launch_tiled_hb<__nv_bfloat16, 8, 8>(hb, grid, smem, st, a);
    }
    return cudaErrorInvalidValue;   // no instance (cannot happen for D <= 256)
}

template <typename E, int RPT, int NF, int KC>
cudaError_t launch_prefill_tiled(const pa_cache_desc* c, int32_t group, int32_t max_q_len,
                                 int32_t num_seqs, cudaStream_t st, const PrefillArgs& a) {
    using Cfg = PrefillTiledCfg<RPT, NF, KC>;
    const int32_t ht = std::min(group, Cfg::kRows), qt = Cfg::kRows / ht;
    const int32_t nsub = (group + ht - 1) / ht;
    if ((int64_t)c->num_kv_heads * nsub > 65535) return cudaErrorInvalidValue;
    const int32_t tiles = std::max(1, (max_q_len + qt - 1) / qt);
    const size_t smem = Cfg::smem_bytes(c->head_dim, elem_bytes(c));
    auto kern = prefill_tiled_kernel<E, RPT, NF, KC>;
    if (!set_smem(kern, smem)) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(tiles, c->num_kv_heads * nsub, num_seqs), dim3(kPtThreads), smem,
                      st, a);
}

// The CUDA-core prefill: 64-row tiles, 32-key chunks up to 128 columns;
// 32-row tiles, 16-key chunks up to 256.
cudaError_t dispatch_prefill_tiled(const pa_cache_desc* c, int32_t group, int32_t max_q_len,
                                   int32_t num_seqs, cudaStream_t st, const PrefillArgs& a) {
    const bool narrow = c->head_dim <= 128;
    if (c->dtype == PA_F32)
        return narrow ? launch_prefill_tiled<float, 4, 4, 32>(c, group, max_q_len, num_seqs, st, a)
                      : launch_prefill_tiled<float, 2, 8, 16>(c, group, max_q_len, num_seqs, st, a);
    return narrow
               ? launch_prefill_tiled<__nv_bfloat16, 4, 4, 32>(c, group, max_q_len, num_seqs, st, a)
               : launch_prefill_tiled<__nv_bfloat16, 2, 8, 16>(c, group, max_q_len, num_seqs, st, a);
}

template <int DMAX, int KC>
cudaError_t launch_prefill_mma(const pa_cache_desc* c, int32_t group, int32_t max_q_len,
                               int32_t num_seqs, cudaStream_t st, const PrefillArgs& a) {
    const int32_t ht = std::min(group, kPmRows), qt = kPmRows / ht;
    const int32_t nsub = (group + ht - 1) / ht;
    if ((int64_t)c->num_kv_heads * nsub > 65535) return cudaErrorInvalidValue;
    const int32_t tiles = std::max(1, (max_q_len + qt - 1) / qt);
    const size_t smem = PrefillMmaCfg<DMAX, KC>::smem_bytes(c->head_dim);
    auto kern = prefill_mma_kernel<DMAX, KC>;
    if (!set_smem(kern, smem)) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(tiles, c->num_kv_heads * nsub, num_seqs), dim3(kPmThreads), smem,
                      st, a);
}

// bf16 head dims that are multiples of 16: the mma.sync prefill, 64-key
// chunks up to 128 columns, 32-key chunks up to 256.
bool prefill_mma_shape(const pa_cache_desc* c) {
    return c->dtype == PA_BF16 && c->head_dim % 16 == 0 && c->head_dim <= 256;
}

cudaError_t dispatch_prefill_mma(const pa_cache_desc* c, int32_t group, int32_t max_q_len,
                                 int32_t num_seqs, cudaStream_t st, const PrefillArgs& a) {
    return c->head_dim <= 128 ? launch_prefill_mma<128, 64>(c, group, max_q_len, num_seqs, st, a)
                              : launch_prefill_mma<256, 32>(c, group, max_q_len, num_seqs, st, a);
}

template <int D, bool CAS>
cudaError_t launch_fast_d(dim3 grid, const CUtensorMap& mk, const CUtensorMap& mv,
                          const DecodeArgs& a, cudaStream_t st) {
    // 16 rows: any CTA may carry 9-16 heads
    return a.group > 8 ? launch_fast<D, true, CAS>(grid, mk, mv, a, st)
                       : launch_fast<D, false, CAS>(grid, mk, mv, a, st);
}

// The shared-prefix instance exists for head dims 64 and 128 only
// (shared_mode() never selects it for the others).
template <bool CAS>
cudaError_t dispatch_fast_cas(dim3 grid, const CUtensorMap& mk, const CUtensorMap& mv,
                              const DecodeArgs& a, cudaStream_t st) {
    switch (a.head_dim) {
        case 64: return launch_fast_d<64, CAS>(grid, mk, mv, a, st);
        case 128: return launch_fast_d<128, CAS>(grid, mk, mv, a, st);
        default: break;
    }
    if constexpr (!CAS) {
        switch (a.head_dim) {
            case 16: return launch_fast_d<16, false>(grid, mk, mv, a, st);
            case 32: return launch_fast_d<32, false>(grid, mk, mv, a, st);
            case 48: return launch_fast_d<48, false>(grid, mk, mv, a, st);
            case 80: return launch_fast_d<80, false>(grid, mk, mv, a, st);
            case 96: return launch_fast_d<96, false>(grid, mk, mv, a, st);
            case 112: return launch_fast_d<112, false>(grid, mk, mv, a, st);
            case 256: return launch_fast_d<256, false>(grid, mk, mv, a, st);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

// cas: the shared-prefix instance (prefix CTAs, members past their shared
// blocks); otherwise the plain decode kernel.
cudaError_t dispatch_fast(dim3 grid, const CUtensorMap& mk, const CUtensorMap& mv,
                          const DecodeArgs& a, cudaStream_t st, bool cas) {
    return cas ? dispatch_fast_cas<true>(grid, mk, mv, a, st)
               : dispatch_fast_cas<false>(grid, mk, mv, a, st);
}

// Address through which kernels reach `p`: device and managed memory as is,
// page-locked host memory through its mapped device pointer.  nullptr for
// pageable host memory (or a null pointer), which a kernel must not touch.
const void* device_view(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return p;
        case cudaMemoryTypeHost:
            return at.devicePointer;
        default:
            return nullptr;
    }
}

// Step arguments (queries, new K/V, slots, tables, lengths, outputs) may be
// device memory or page-locked host memory; the kernels then read or write
// the host memory directly over the host link (NVLink-C2C on Grace-Blackwell),
// with no staging copy.  Replaces p by the address kernels use; false for
// pageable host memory, which a kernel must never touch.
template <typename T>
bool map_step_arg(T*& p) {
    if (!p) return true;
    const void* view = device_view(p);
    if (!view) return false;
    p = static_cast<T*>(const_cast<void*>(view));
    return true;
}

// Caches and workspaces: device (or managed) memory only.
bool device_memory(const void* p) {
    if (!p) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Launch the cache-write kernel with the widest vector the row size and the
// pointers' alignment allow.
template <typename SlotFn>
pa_status launch_write(const void* k, const void* v, SlotFn slot_of, int32_t num_tokens,
                       void* k_cache, void* v_cache, const pa_cache_desc* cache,
                       cudaStream_t st) {
    if (!k || !v || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!map_step_arg(k) || !map_step_arg(v) || !device_memory(k_cache) ||
        !device_memory(v_cache))
        return PA_ERR_INVALID_ARG;
    const int32_t row = cache->head_dim * elem_bytes(cache);
    int vec = 16;
    while (vec > 2 && (row % vec || !aligned(k, vec) || !aligned(v, vec) ||
                       !aligned(k_cache, vec) || !aligned(v_cache, vec)))
        vec >>= 1;
    if (row % vec || !aligned(k, vec) || !aligned(v, vec) || !aligned(k_cache, vec) ||
        !aligned(v_cache, vec))
        return PA_ERR_INVALID_ARG;
    // one warp per token (kWriteWarps tokens a CTA), at most 16 CTAs per SM
    // with a grid-stride loop past that
    const int threads = 32 * kWriteWarps;
    const int64_t sms = std::max(1, device_sm_count());
    const unsigned blocks = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>(((int64_t)num_tokens + kWriteWarps - 1) / kWriteWarps, sms * 16));
    const int64_t num_slots = (int64_t)cache->num_blocks * cache->block_size;
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3(blocks), dim3(threads), 0, st,
                          static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(v), slot_of,
                          (int64_t)num_tokens, static_cast<uint8_t*>(k_cache),
                          static_cast<uint8_t*>(v_cache), cache->num_kv_heads,
                          cache->block_size, num_slots, row);
    };
    cudaError_t err;
    switch (vec) {
        case 16: err = go(write_kv_kernel<16, SlotFn>); break;
        case 8: err = go(write_kv_kernel<8, SlotFn>); break;
        case 4: err = go(write_kv_kernel<4, SlotFn>); break;
        default: err = go(write_kv_kernel<2, SlotFn>); break;
    }
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// An NVTX range over one library call (host side: argument checks and
// launches), so profilers can attribute the kernels to the call that made them.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

}  // namespace
}  // namespace pa

using namespace pa;

namespace pa {
namespace {

// Groups of a shared-prefix decode call (host view of its arguments).
struct ShareGroups {
    const int32_t* seq_group;
    const int32_t* member_start;
    const int32_t* members;
    const int32_t* prefix_blocks;
    int32_t num_groups, max_group_size, max_prefix_blocks;
    int32_t mode;   // pa_shared_mode
};

// Workspace slots per (sequence, head) of a shared-prefix call: the longest
// shared prefix's partitions, then the longest sequence's own.
int64_t cascade_slots(int32_t max_seq_len, int32_t max_prefix_blocks, int32_t part,
                      const pa_cache_desc* c) {
    return ((int64_t)max_prefix_blocks * c->block_size + part - 1) / part +
           num_parts(max_seq_len, part);
}

// Whether a shared-prefix call reads the shared blocks once per row tile
// (1) or runs the plain decode over the same tables (0); < 0 for invalid
// arguments.  Automatic: once when a row tile holds m >= 2 members (m = 8
// or 16 rows / query heads per kv head) and the shared prefix saves
// tokens * (1 - 1/m) >= PA_SHARED_MIN_SAVED tokens of reads per member.
// Measured on GQA-shaped batches (per call, shared / plain): G = 4 with a
// 512-token prefix (m = 2, 256 saved) 0.985; 2048 tokens (1024) 1.007; 4096
// tokens and 64 members 1.156; G = 1 with 2048 tokens (m = 8) 1.21; G = 8
// (m = 1) 0.87.  Below the threshold the members' extra merges cost more than
// the shared reads, which the plain decode takes from L2, save.
#ifndef PA_SHARED_MIN_SAVED
#define PA_SHARED_MIN_SAVED 1024
#endif
int32_t shared_mode(int32_t num_q_heads, int32_t max_prefix_blocks, int32_t mode,
                    const pa_cache_desc* c) {
    if (!desc_ok(c) || num_q_heads <= 0 || num_q_heads % c->num_kv_heads ||
        max_prefix_blocks < 0 || mode < PA_SHARED_AUTO || mode > PA_SHARED_PLAIN)
        return -1;
    const int32_t group = num_q_heads / c->num_kv_heads;
    if (!fast_shape(c, group) || (c->head_dim != 64 && c->head_dim != 128) ||
        mode == PA_SHARED_PLAIN)
        return 0;
    if (mode == PA_SHARED_ONCE) return 1;
    const int64_t rows = group > 8 ? 16 : 8;
    const int64_t m = rows / group;                       // members per row tile
    if (m < 2) return 0;
    const int64_t saved = (int64_t)max_prefix_blocks * c->block_size * (m - 1) / m;
    return saved >= PA_SHARED_MIN_SAVED ? 1 : 0;
}

// Bytes of `cells` workspace cells: acc (head_dim floats) then (m, l).
size_t cells_bytes(size_t cells, const pa_cache_desc* c) {
    return align256(cells * c->head_dim * sizeof(float)) + align256(cells * 2 * sizeof(float));
}

// pa_decode, and with `sh` (groups sharing leading blocks) the shared-prefix
// decode: on the TMA kernel, extra CTAs attend each group's shared blocks once
// for all its members' query heads, members' own CTAs start past them, and
// the merge combines both.  Other kernels run the plain decode over the same
// tables (same result).
//
// With k_new / v_new (a decode step's append, never with `sh`), sequence i's
// token at position seq_lens[i] - 1 is first written to the caches: inside
// the TMA kernel (the CTA holding that position uses the new rows in place of
// the slot's old contents and stores them), else by the cache-write kernel
// with slots from the lengths, launched before the decode.
pa_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                      const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                      int32_t num_q_heads, float scale, int32_t partition_tokens, void* out,
                      void* workspace, size_t workspace_bytes_given, const pa_cache_desc* cache,
                      void* stream, const ShareGroups* sh, const void* k_new = nullptr,
                      const void* v_new = nullptr) {
    const int32_t path = !desc_ok(cache) || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads
                             ? -1
                             : fast_shape(cache, num_q_heads / cache->num_kv_heads) ? 1
                             : mma_shape(cache, num_q_heads / cache->num_kv_heads)  ? 2
                                                                                    : 0;
    if (path < 0 || num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq < 0 ||
        partition_tokens < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
        return PA_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * cache->block_size < max_seq_len) return PA_ERR_INVALID_ARG;
    if (num_seqs > 65535 || cache->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    const int32_t group = num_q_heads / cache->num_kv_heads;
    const int32_t B = cache->block_size;
    int32_t part = partition_tokens ? partition_tokens
                                    : auto_partition(num_seqs, num_q_heads, max_seq_len, cache);
    if (part <= 0 || part % B) return PA_ERR_INVALID_ARG;
    bool fast = path == 1;
    if (fast && (part > fast_max_partition(cache) || !aligned(k_cache, 16) ||
                 !aligned(v_cache, 16) || !aligned(q, 16)))
        fast = false;
    // other shapes: the mma.sync kernel (bf16, head dims that are multiples of
    // 16 up to 128), the tiled CUDA-core kernel, else (a head dim that is not
    // whole 16-byte rows, or unaligned caches) the generic one
    const bool caches16 = aligned(k_cache, 16) && aligned(v_cache, 16);
    const bool mma = path == 2 && caches16 && aligned(q, 4);
    const bool tiled = !fast && !mma && tiled_shape(cache) && caches16;
    if (!fast && !mma && !tiled && part > generic_max_partition(cache, group))
        return PA_ERR_UNSUPPORTED;
    if (!aligned(q, elem_bytes(cache)) || !aligned(out, elem_bytes(cache)) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!map_step_arg(q) || !map_step_arg(block_tables) || !map_step_arg(seq_lens) ||
        !map_step_arg(out) || !device_memory(k_cache) || !device_memory(v_cache))
        return PA_ERR_INVALID_ARG;
    if (num_parts(max_seq_len, part) > 65535) return PA_ERR_UNSUPPORTED;
    // the append: fused into the TMA kernel when its 16-byte row pieces are
    // aligned, else a separate cache write first
    const bool append = k_new != nullptr || v_new != nullptr;
    if (append && (!k_new || !v_new || sh || !aligned(k_new, elem_bytes(cache)) ||
                   !aligned(v_new, elem_bytes(cache)) || !map_step_arg(k_new) ||
                   !map_step_arg(v_new)))
        return PA_ERR_INVALID_ARG;
    // (the kernel's row patch covers 128 columns: head dim 256 writes first)
    const bool fused = append && fast && cache->head_dim <= 128 && aligned(k_new, 16) &&
                       aligned(v_new, 16);
    // shared-prefix decode on the TMA kernel: workspace slots for the
    // groups' prefix partitions in front of each member's own
    const bool cas = sh != nullptr && fast &&
                     shared_mode(num_q_heads, sh->max_prefix_blocks, sh->mode, cache) == 1;
    const int64_t slots = cas ? cascade_slots(max_seq_len, sh->max_prefix_blocks, part, cache)
                              : num_parts(max_seq_len, part);
    if (slots > 65535) return PA_ERR_UNSUPPORTED;
    const int32_t max_parts = (int32_t)slots;
    const size_t need = cas ? cells_bytes((size_t)num_seqs * num_q_heads * slots, cache)
                            : workspace_bytes(num_seqs, num_q_heads, max_seq_len, part, cache);
    if (need > 0 && (!workspace || workspace_bytes_given < need || !aligned(workspace, 256) ||
                     !device_memory(workspace)))
        return PA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug::enabled()) {
        const pa_status r = debug::check_tables(block_tables, max_blocks_per_seq, seq_lens,
                                                num_seqs, max_seq_len, nullptr, 0, cache, st);
        if (r != PA_OK) return r;
        if (append) {
            const pa_status r3 = debug::check_appends(block_tables, max_blocks_per_seq, seq_lens,
                                                      num_seqs, cache, st);
            if (r3 != PA_OK) return r3;
        }
        if (sh) {
            const pa_status r2 = debug::check_groups(block_tables, max_blocks_per_seq, num_seqs,
                                                     sh->seq_group, sh->member_start,
                                                     sh->members, sh->prefix_blocks,
                                                     sh->num_groups, sh->max_group_size,
                                                     sh->max_prefix_blocks, st);
            if (r2 != PA_OK) return r2;
        }
    }

    DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    const size_t cells = (size_t)num_seqs * num_q_heads * max_parts;
    a.ws_acc = need ? static_cast<float*>(workspace) : nullptr;
    a.ws_ml = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              align256(cells * cache->head_dim * sizeof(float)))
                   : nullptr;
    a.num_seqs = num_seqs;
    a.max_blocks = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = cache->num_kv_heads;
    a.group = group;
    a.num_blocks = cache->num_blocks;
    a.block_size = B;
    a.head_dim = cache->head_dim;
    a.part_tokens = part;
    a.max_parts = max_parts;
    a.scale_log2 = scale * kLog2e;
    a.sub_groups = fast || mma ? (group + 15) / 16
                   : tiled     ? (group + kTiledHeads - 1) / kTiledHeads
                               : 1;
    if ((int64_t)cache->num_kv_heads * a.sub_groups > 65535) return PA_ERR_UNSUPPORTED;

    dim3 grid(max_parts, cache->num_kv_heads * a.sub_groups, num_seqs);
    if (cas) {
        // prefix CTAs: per group, tiles of kRows (member, head) rows, spread
        // over the sub-group index and prefix_ztiles grid z slots
        const int64_t rows = group > 8 ? 16 : 8;
        const int64_t tiles = ((int64_t)sh->max_group_size * group + rows - 1) / rows;
        const int64_t zt = (tiles + a.sub_groups - 1) / a.sub_groups;
        const int64_t pz = zt * sh->num_groups;
        if (pz + num_seqs > 65535) return PA_ERR_UNSUPPORTED;
        a.seq_group = sh->seq_group;
        a.member_start = sh->member_start;
        a.members = sh->members;
        a.prefix_blocks = sh->prefix_blocks;
        a.num_groups = sh->num_groups;
        a.max_group_size = sh->max_group_size;
        a.max_prefix_blocks = sh->max_prefix_blocks;
        a.prefix_ztiles = (int32_t)zt;
        a.prefix_z = (int32_t)pz;
        const int64_t own = num_parts(max_seq_len, part);
        const int64_t pre = ((int64_t)sh->max_prefix_blocks * B + part - 1) / part;
        grid = dim3((unsigned)std::max(own, pre), cache->num_kv_heads * a.sub_groups,
                    (unsigned)(pz + num_seqs));
    }
    if (fused) {
        a.k_new = k_new;
        a.v_new = v_new;
    } else if (append) {
        const SlotFromAppend slots{seq_lens, block_tables, max_blocks_per_seq, B,
                                   cache->num_blocks, max_seq_len};
        const pa_status w = launch_write(k_new, v_new, slots, num_seqs, const_cast<void*>(k_cache),
                                         const_cast<void*>(v_cache), cache, st);
        if (w != PA_OK) return w;
    }
    cudaError_t err;
    if (fast) {
        CUtensorMap mk, mv;
        if (!cached_map(&mk, k_cache, cache, 0) || !cached_map(&mv, v_cache, cache, 1))
            return PA_ERR_CUDA;
        err = dispatch_fast(grid, mk, mv, a, st, cas);
    } else if (mma) {
        const size_t smem = decode_mma_smem_bytes(cache->head_dim);
        auto kern = group > 8 ? decode_mma_kernel<true> : decode_mma_kernel<false>;
        if (!set_smem(kern, smem)) return PA_ERR_UNSUPPORTED;
        err = launch_pdl(kern, grid, dim3(kMmaThreads), smem, st, a);
    } else if (tiled) {
        err = dispatch_tiled(cache, group, grid, a, st);
        if (err == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
    } else {
        const size_t smem = generic_smem_bytes(group, cache->head_dim, part, B);
        if (cache->dtype == PA_F32) {
            if (!set_smem(decode_generic_kernel<float>, smem)) return PA_ERR_UNSUPPORTED;
            err = launch_pdl(decode_generic_kernel<float>, grid, dim3(128), smem, st, a);
        } else {
            if (!set_smem(decode_generic_kernel<__nv_bfloat16>, smem)) return PA_ERR_UNSUPPORTED;
            err = launch_pdl(decode_generic_kernel<__nv_bfloat16>, grid, dim3(128), smem, st, a);
        }
    }
    if (err != cudaSuccess) return PA_ERR_CUDA;
    if (max_parts > 1 || cas) {
        // the longest sequence's own partitions (a shared-prefix call's extra
        // prefix slots are mostly one or two per member)
        const int32_t typical = (int32_t)num_parts(max_seq_len, part);
        const cudaError_t merr = cache->dtype == PA_F32
                                     ? launch_merge<float>(a, st, typical)
                                     : launch_merge<__nv_bfloat16>(a, st, typical);
        if (merr != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache,
                      const pa_cache_desc* cache, void* stream) {
    const CallRange range("pa_write_kv");
    if (!desc_ok(cache) || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!slot_mapping || !aligned(slot_mapping, 8) || !map_step_arg(slot_mapping))
        return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug::enabled()) {
        const pa_status r = debug::check_slots(
            slot_mapping, num_tokens, (int64_t)cache->num_blocks * cache->block_size, st);
        if (r != PA_OK) return r;
    }
    return launch_write(k, v, SlotFromMapping{slot_mapping}, num_tokens, k_cache, v_cache, cache,
                        st);
}

pa_status pa_write_kv_positions(const void* k, const void* v, const int32_t* seq_ids,
                                const int32_t* positions, int32_t num_tokens,
                                const int32_t* block_tables, int32_t num_seqs,
                                int32_t max_blocks_per_seq, void* k_cache, void* v_cache,
                                const pa_cache_desc* cache, void* stream) {
    const CallRange range("pa_write_kv_positions");
    if (!desc_ok(cache) || num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!seq_ids || !positions || !block_tables || !aligned(seq_ids, 4) ||
        !aligned(positions, 4) || !aligned(block_tables, 4))
        return PA_ERR_INVALID_ARG;
    if (!map_step_arg(seq_ids) || !map_step_arg(positions) || !map_step_arg(block_tables))
        return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug::enabled()) {
        const pa_status r = debug::check_positions(seq_ids, positions, num_tokens, block_tables,
                                                   num_seqs, max_blocks_per_seq, cache, st);
        if (r != PA_OK) return r;
    }
    SlotFromPosition fn{seq_ids, positions, block_tables, num_seqs, max_blocks_per_seq,
                        cache->block_size, cache->num_blocks};
    return launch_write(k, v, fn, num_tokens, k_cache, v_cache, cache, st);
}

pa_status pa_copy_blocks(const void* src_k, const void* src_v, int32_t src_num_blocks,
                         void* dst_k, void* dst_v, int32_t dst_num_blocks,
                         const int64_t* block_pairs, int32_t num_pairs,
                         const pa_cache_desc* cache, void* stream) {
    const CallRange range("pa_copy_blocks");
    if (!desc_ok(cache) || num_pairs < 0 || src_num_blocks < 0 || dst_num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    const void* sk = device_view(src_k);
    const void* sv = device_view(src_v);
    void* dk = const_cast<void*>(device_view(dst_k));
    void* dv = const_cast<void*>(device_view(dst_v));
    const int64_t* pairs = static_cast<const int64_t*>(device_view(block_pairs));
    if (!sk || !sv || !dk || !dv || !pairs || !aligned(pairs, 8)) return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)cache->num_kv_heads * cache->block_size *
                                cache->head_dim * elem_bytes(cache);
    int vec = 16;
    while (vec > 2 && (block_bytes % vec || !aligned(sk, vec) || !aligned(sv, vec) ||
                       !aligned(dk, vec) || !aligned(dv, vec)))
        vec >>= 1;
    if (block_bytes % vec || !aligned(sk, vec) || !aligned(sv, vec) || !aligned(dk, vec) ||
        !aligned(dv, vec))
        return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug::enabled()) {
        const pa_status r = debug::check_pairs(pairs, num_pairs, src_num_blocks, dst_num_blocks,
                                               sk == dk, st);
        if (r != PA_OK) return r;
    }
    const int64_t total = (int64_t)num_pairs * 2 * (block_bytes / vec);
    const int threads = 256;
    const int64_t sms = std::max(1, device_sm_count());
    const unsigned blocks = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>((total + threads - 1) / threads, sms * 16));
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3(blocks), dim3(threads), 0, st,
                          static_cast<const uint8_t*>(sk), static_cast<const uint8_t*>(sv),
                          (int64_t)src_num_blocks, static_cast<uint8_t*>(dk),
                          static_cast<uint8_t*>(dv), (int64_t)dst_num_blocks, pairs,
                          (int64_t)num_pairs, block_bytes);
    };
    cudaError_t err;
    switch (vec) {
        case 16: err = go(copy_blocks_kernel<16>); break;
        case 8: err = go(copy_blocks_kernel<8>); break;
        case 4: err = go(copy_blocks_kernel<4>); break;
        default: err = go(copy_blocks_kernel<2>); break;
    }
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int32_t pa_decode_path(int32_t num_q_heads, const pa_cache_desc* cache) {
    if (!desc_ok(cache) || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return -1;
    const int32_t group = num_q_heads / cache->num_kv_heads;
    return fast_shape(cache, group) ? 1 : mma_shape(cache, group) ? 2 : 0;
}

int32_t pa_decode_partition_tokens(int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                                   const pa_cache_desc* cache) {
    if (pa_decode_path(num_q_heads, cache) < 0 || num_seqs < 0 || max_seq_len < 0) return -1;
    return auto_partition(num_seqs, num_q_heads, max_seq_len, cache);
}

size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                                 int32_t partition_tokens, const pa_cache_desc* cache) {
    if (pa_decode_path(num_q_heads, cache) < 0 || num_seqs < 0 || max_seq_len < 0) return 0;
    const int32_t part = partition_tokens > 0
                             ? partition_tokens
                             : auto_partition(num_seqs, num_q_heads, max_seq_len, cache);
    return workspace_bytes(num_seqs, num_q_heads, max_seq_len, part, cache);
}

pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_q_heads, float scale, int32_t partition_tokens, void* out,
                    void* workspace, size_t workspace_bytes_given, const pa_cache_desc* cache,
                    void* stream) {
    const CallRange range("pa_decode");
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, max_seq_len, num_q_heads, scale, partition_tokens, out,
                       workspace, workspace_bytes_given, cache, stream, nullptr);
}

pa_status pa_decode_append(const void* q, const void* k_new, const void* v_new, void* k_cache,
                           void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                           int32_t num_q_heads, float scale, int32_t partition_tokens, void* out,
                           void* workspace, size_t workspace_bytes_given,
                           const pa_cache_desc* cache, void* stream) {
    const CallRange range("pa_decode_append");
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, max_seq_len, num_q_heads, scale, partition_tokens, out,
                       workspace, workspace_bytes_given, cache, stream, nullptr, k_new, v_new);
}

int32_t pa_decode_shared_prefix_mode(int32_t num_q_heads, int32_t max_prefix_blocks,
                                     int32_t mode, const pa_cache_desc* cache) {
    return shared_mode(num_q_heads, max_prefix_blocks, mode, cache);
}

size_t pa_decode_shared_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                               int32_t max_seq_len, int32_t max_prefix_blocks,
                                               int32_t partition_tokens,
                                               const pa_cache_desc* cache) {
    if (pa_decode_path(num_q_heads, cache) < 0 || num_seqs < 0 || max_seq_len < 0 ||
        max_prefix_blocks < 0 || partition_tokens < 0)
        return 0;
    const int32_t part = partition_tokens > 0
                             ? partition_tokens
                             : auto_partition(num_seqs, num_q_heads, max_seq_len, cache);
    if (part <= 0) return 0;
    const size_t plain = workspace_bytes(num_seqs, num_q_heads, max_seq_len, part, cache);
    if (shared_mode(num_q_heads, max_prefix_blocks, PA_SHARED_ONCE, cache) != 1) return plain;
    const int64_t slots = cascade_slots(max_seq_len, max_prefix_blocks, part, cache);
    return std::max(plain, cells_bytes((size_t)num_seqs * num_q_heads * slots, cache));
}

pa_status pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs,
                                  int32_t max_seq_len, int32_t num_q_heads, float scale,
                                  int32_t partition_tokens, const int32_t* seq_group,
                                  const int32_t* member_start, const int32_t* members,
                                  const int32_t* prefix_blocks, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_blocks,
                                  int32_t mode, void* out, void* workspace,
                                  size_t workspace_bytes_given, const pa_cache_desc* cache,
                                  void* stream) {
    const CallRange range("pa_decode_shared_prefix");
    if (num_groups < 0 || max_group_size < 0 || max_prefix_blocks < 0 ||
        max_prefix_blocks > max_blocks_per_seq || mode < PA_SHARED_AUTO ||
        mode > PA_SHARED_PLAIN)
        return PA_ERR_INVALID_ARG;
    if (num_groups == 0)
        return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                           num_seqs, max_seq_len, num_q_heads, scale, partition_tokens, out,
                           workspace, workspace_bytes_given, cache, stream, nullptr);
    if (!seq_group || !member_start || !members || !prefix_blocks || max_group_size < 1)
        return PA_ERR_INVALID_ARG;
    if (!aligned(seq_group, 4) || !aligned(member_start, 4) || !aligned(members, 4) ||
        !aligned(prefix_blocks, 4))
        return PA_ERR_INVALID_ARG;
    if (!map_step_arg(seq_group) || !map_step_arg(member_start) || !map_step_arg(members) ||
        !map_step_arg(prefix_blocks))
        return PA_ERR_INVALID_ARG;
    ShareGroups sh;
    sh.seq_group = seq_group;
    sh.member_start = member_start;
    sh.members = members;
    sh.prefix_blocks = prefix_blocks;
    sh.num_groups = num_groups;
    sh.max_group_size = max_group_size;
    sh.max_prefix_blocks = max_prefix_blocks;
    sh.mode = mode;
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, max_seq_len, num_q_heads, scale, partition_tokens, out,
                       workspace, workspace_bytes_given, cache, stream, &sh);
}

pa_status pa_prefill(const void* q, const int32_t* query_start_loc, int32_t total_q,
                     int32_t max_q_len, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                     int32_t num_q_heads, float scale, void* out, const pa_cache_desc* cache,
                     void* stream) {
    const CallRange range("pa_prefill");
    const int32_t path = pa_decode_path(num_q_heads, cache);
    if (path < 0 || num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_seq_len < 0 ||
        max_blocks_per_seq < 0 || max_q_len > max_seq_len)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    if (!q || !query_start_loc || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
        return PA_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * cache->block_size < max_seq_len) return PA_ERR_INVALID_ARG;
    if (num_seqs > 65535 || cache->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    const int32_t group = num_q_heads / cache->num_kv_heads;
    const int eb = elem_bytes(cache);
    if (!aligned(q, eb) || !aligned(out, eb) || !aligned(query_start_loc, 4) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!map_step_arg(q) || !map_step_arg(query_start_loc) || !map_step_arg(block_tables) ||
        !map_step_arg(seq_lens) || !map_step_arg(out) || !device_memory(k_cache) ||
        !device_memory(v_cache))
        return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug::enabled()) {
        const pa_status r = debug::check_tables(block_tables, max_blocks_per_seq, seq_lens,
                                                num_seqs, max_seq_len, query_start_loc, total_q,
                                                cache, st);
        if (r != PA_OK) return r;
    }
    PrefillArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.query_start = query_start_loc;
    a.seq_lens = seq_lens;
    a.block_tables = block_tables;
    a.out = out;
    a.num_seqs = num_seqs;
    a.max_blocks = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = cache->num_kv_heads;
    a.group = group;
    a.num_blocks = cache->num_blocks;
    a.block_size = cache->block_size;
    a.head_dim = cache->head_dim;
    // 128-row tcgen05 tiles of floor(128 / G) tokens x G heads (the last
    // 128 mod G rows idle)
    a.tokens_per_tile = group <= 128 ? 128 / group : 0;
    constexpr int32_t kTilesPerCta = 2;
    a.scale_log2 = scale * kLog2e;
    // the tensor-core kernel takes its row maximum before scaling: scale >= 0
    // (head dims 16-48 run in a 64-column tile, 80-112 in a 128-column one,
    // whose columns past the head dim are zeros)
    const bool fast = path == 1 && cache->head_dim <= 128 && a.tokens_per_tile > 0 &&
                      aligned(q, 16) && aligned(out, 16) && aligned(k_cache, 16) &&
                      aligned(v_cache, 16) && scale >= 0.f;
    cudaError_t err;
    if (fast) {
        CUtensorMap mk, mv;
        if (!cached_map(&mk, k_cache, cache, 0) || !cached_map(&mv, v_cache, cache, 1))
            return PA_ERR_CUDA;
        const int32_t per_cta = kTilesPerCta * a.tokens_per_tile;
        const int32_t tiles = std::max(1, (max_q_len + per_cta - 1) / per_cta);
        dim3 grid(tiles, cache->num_kv_heads, num_seqs);
        if (cache->head_dim > 64) {
            using Cfg = PrefillWsCfg<128, PA_PREFILL_KEYS>;
            auto kern = prefill_ws_kernel<128, PA_PREFILL_KEYS>;
            if (!set_smem(kern, Cfg::smem_bytes())) return PA_ERR_UNSUPPORTED;
            err = launch_pdl(kern, grid, dim3(Cfg::kThreads), Cfg::smem_bytes(), st, mk, mv, a);
        } else {
            using Cfg = PrefillWsCfg<64, PA_PREFILL_KEYS>;
            auto kern = prefill_ws_kernel<64, PA_PREFILL_KEYS>;
            if (!set_smem(kern, Cfg::smem_bytes())) return PA_ERR_UNSUPPORTED;
            err = launch_pdl(kern, grid, dim3(Cfg::kThreads), Cfg::smem_bytes(), st, mk, mv, a);
        }
    } else if (prefill_mma_shape(cache) && aligned(q, 16) && aligned(out, 4) &&
               aligned(k_cache, 16) && aligned(v_cache, 16)) {
        err = dispatch_prefill_mma(cache, group, max_q_len, num_seqs, st, a);
        if (err == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
    } else if (tiled_shape(cache) && aligned(k_cache, 16) && aligned(v_cache, 16) &&
               aligned(out, 16)) {
        // (the output is stored four values at a time)
        err = dispatch_prefill_tiled(cache, group, max_q_len, num_seqs, st, a);
        if (err == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
    } else {
        if (cache->head_dim > 32 * kGenericMaxDimPerLane) return PA_ERR_UNSUPPORTED;
        dim3 grid(total_q, cache->num_kv_heads);
        if (cache->dtype == PA_F32)
            err = launch_pdl(prefill_generic_kernel<float>, grid, dim3(128), 0, st, a);
        else
            err = launch_pdl(prefill_generic_kernel<__nv_bfloat16>, grid, dim3(128), 0, st, a);
    }
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

const char* pa_status_str(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or size";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

pa_status pa_check_wait_timeout(int32_t expected, int32_t arrivals, int64_t limit_cycles,
                                void* stream) {
    if (expected < 1 || expected > 1024 || arrivals < 0 || arrivals > expected ||
        limit_cycles < 1000 || limit_cycles > (1LL << 31))
        return PA_ERR_INVALID_ARG;
    const int32_t threads = ((std::max(32, expected) + 31) / 32) * 32;
    pa::wait_check_kernel<<<1, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        expected, arrivals, (long long)limit_cycles);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int32_t pa_last_device_error(void) {
    unsigned int bits = 0, zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(&bits, pa::g_device_error, sizeof(bits)) != cudaSuccess) return -1;
    if (cudaMemcpyToSymbol(pa::g_device_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return (int32_t)bits;
}

}  // extern "C"

// ---- decode without any caller-provided workspace -------------------------------
//
// Some callers cannot allocate device memory at the point where they run
// attention: a plugin hook of an inference engine that forbids allocation once
// execution has started, or a process with a fixed, pre-reserved memory budget
// that has no room to grow.  pa_decode_no_alloc serves them by keeping the
// split-K workspace in a fixed array inside the library itself.  The array is
// a file-scope device variable, so every GPU that loads libpa.so holds it
// until the process exits.  In host code the name g_no_alloc_workspace is
// only a host-side stand-in, not a device address: the real address is looked
// up with cudaGetSymbolAddress, with the device current, and cached per device
// together with the id of the context it was found in.  A later call whose
// current context differs (the device was reset, so the module was loaded
// again and the array may have moved) looks it up again.

static __device__ __align__(256) unsigned char g_no_alloc_workspace[PA_NO_ALLOC_WORKSPACE_BYTES];

namespace pa {
namespace {

struct NoAllocEntry {
    void* ptr = nullptr;
    unsigned long long ctx = 0;   // cuCtxGetId of the context ptr belongs to
};
NoAllocEntry g_no_alloc[kMaxDevices];
std::mutex g_no_alloc_mutex;

// Id of the calling thread's current context, 0 when none is current yet or
// the driver entry points are unavailable.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the static workspace for the current device, or nullptr
// if the lookup failed.  Runs cudaGetSymbolAddress on the first use per device
// and again whenever the current context is not the one the cached address
// came from (or cannot be identified).
void* no_alloc_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_no_alloc_mutex);
    NoAllocEntry& e = g_no_alloc[dev];
    const unsigned long long ctx = current_context_id();
    if (e.ptr == nullptr || ctx == 0 || ctx != e.ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_workspace) != cudaSuccess) return nullptr;
        e.ptr = p;
        e.ctx = current_context_id();   // the lookup made the device's context current
    }
    return e.ptr;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, int32_t num_seqs,
                                        int32_t max_seq_len, int32_t num_q_heads, float scale,
                                        int32_t partition_tokens, void* out,
                                        const pa_cache_desc* cache, void* stream) {
    if (pa_decode_path(num_q_heads, cache) < 0 || num_seqs < 0 || max_seq_len < 0 ||
        partition_tokens < 0)
        return PA_ERR_INVALID_ARG;
    // the partition count first: a request pa_decode would refuse for it is
    // refused the same way here, before the workspace is sized
    const int32_t part = partition_tokens > 0
                             ? partition_tokens
                             : pa::auto_partition(num_seqs, num_q_heads, max_seq_len, cache);
    if (part <= 0) return PA_ERR_INVALID_ARG;
    if (pa::num_parts(max_seq_len, part) > 65535) return PA_ERR_UNSUPPORTED;
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, max_seq_len,
                                                  partition_tokens, cache);
    if (need > PA_NO_ALLOC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
    void* ws = pa::no_alloc_workspace();
    if (ws == nullptr) return PA_ERR_CUDA;
    return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     max_seq_len, num_q_heads, scale, partition_tokens, out, ws,
                     PA_NO_ALLOC_WORKSPACE_BYTES, cache, stream);
}
