// pa.cu -- C-ABI entry points of libpa.so (declared in include/pa.h).
//
// Host side only: argument checks, kernel selection, split-K sizing, TMA
// descriptor encoding and launches on the caller's stream.  Every step of the
// computation runs in the kernels of the included headers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "decode_generic.cuh"
#include "decode_tma_mma.cuh"
#include "merge.cuh"
#include "write_kv.cuh"

#ifndef PA_USE_PDL
#define PA_USE_PDL 1   // launch with programmatic stream serialization
#endif
#ifndef PA_TARGET_CTAS_PER_SM
#define PA_TARGET_CTAS_PER_SM 8
#endif
#ifndef PA_MAX_PARTITION_TOKENS
#define PA_MAX_PARTITION_TOKENS 1024
#endif

namespace pa {
namespace {

constexpr int kMaxDevices = 64;

int device_sm_count() {
    static int cached[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

bool desc_ok(const pa_cache_desc* c) {
    return c && c->num_blocks > 0 && c->block_size > 0 && c->num_kv_heads > 0 &&
           c->head_dim > 0 && (c->dtype == PA_F32 || c->dtype == PA_BF16);
}

int elem_bytes(const pa_cache_desc* c) { return c->dtype == PA_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- kernel selection --------------------------------------------------------

bool fast_shape(const pa_cache_desc* c, int32_t group) {
    if (c->dtype != PA_BF16 || group < 1 || group > 16) return false;
    const int D = c->head_dim, B = c->block_size;
    if (D != 64 && D != 128) return false;
    return B % 16 == 0 && B <= 256;
}

// Largest partition (tokens) the generic kernel's shared memory holds.
int32_t generic_max_partition(const pa_cache_desc* c, int32_t group) {
    const size_t budget = 96 * 1024;
    int32_t B = c->block_size;
    int64_t fixed = 4LL * ((int64_t)group * c->head_dim + 2 * group);
    int64_t per_tok = 4LL * group;
    int64_t p = (int64_t(budget) - fixed) / per_tok;
    p = p / B * B;
    return (int32_t)std::max<int64_t>(p, 0);
}

int32_t fast_max_partition(const pa_cache_desc* c) {
    return 2048 * c->block_size;   // TmaMmaCfg::kMaxTableSlice blocks
}

int32_t auto_partition(int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                       const pa_cache_desc* c) {
    const int32_t B = c->block_size;
    const int32_t group = num_q_heads / c->num_kv_heads;
    if (!fast_shape(c, group)) {
        int32_t cap = generic_max_partition(c, group);
        int32_t want = std::max(B, (512 / B) * B);
        return std::max(B, std::min(cap, want));
    }
    // one block per warp per step; aim for about PA_TARGET_CTAS_PER_SM CTAs
    // per SM over the batch (counted at max_seq_len), between 4 blocks and
    // PA_MAX_PARTITION_TOKENS tokens
    const int64_t unit = 4LL * B;
    const int64_t sms = std::max(1, device_sm_count());
    const int64_t work = (int64_t)num_seqs * c->num_kv_heads * std::max(max_seq_len, 1);
    const int64_t target = (int64_t)PA_TARGET_CTAS_PER_SM * sms;
    int64_t p = (work + target - 1) / target;
    p = (p + unit - 1) / unit * unit;
    const int64_t cap = std::max<int64_t>(unit, PA_MAX_PARTITION_TOKENS / unit * unit);
    p = std::min(std::max(p, unit), cap);
    p = std::min<int64_t>(p, fast_max_partition(c));
    return (int32_t)p;
}

int32_t num_parts(int32_t max_seq_len, int32_t part) {
    return std::max(1, (max_seq_len + part - 1) / part);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                       int32_t part, const pa_cache_desc* c) {
    const int32_t P = num_parts(max_seq_len, part);
    if (P <= 1) return 0;
    const size_t cells = (size_t)num_seqs * num_q_heads * P;
    return align256(cells * c->head_dim * sizeof(float)) + align256(cells * 2 * sizeof(float));
}

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
    cuuint32_t box[3] = {64, 16, 1};
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

template <typename Kern>
bool set_smem(Kern kern, size_t bytes) {
    if (bytes <= 48 * 1024) return true;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)bytes) == cudaSuccess;
}

template <int D, bool G16>
cudaError_t launch_fast(dim3 grid, const CUtensorMap& mk, const CUtensorMap& mv,
                        const DecodeArgs& a, cudaStream_t st) {
    using C = TmaMmaCfg<D, G16>;
    auto kern = decode_tma_mma_kernel<D, G16>;
    if (!set_smem(kern, C::smem_bytes_max())) return cudaErrorInvalidValue;
    const size_t smem = C::smem_bytes(a.part_tokens, a.block_size);
    return launch_pdl(kern, grid, dim3(C::kThreads), smem, st, mk, mv, a);
}

cudaError_t dispatch_fast(dim3 grid, const CUtensorMap& mk, const CUtensorMap& mv,
                          const DecodeArgs& a, cudaStream_t st) {
    const bool g16 = a.group > 8;
    switch (a.head_dim) {
        case 64: return g16 ? launch_fast<64, true>(grid, mk, mv, a, st)
                            : launch_fast<64, false>(grid, mk, mv, a, st);
        case 128: return g16 ? launch_fast<128, true>(grid, mk, mv, a, st)
                             : launch_fast<128, false>(grid, mk, mv, a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache,
                      const pa_cache_desc* cache, void* stream) {
    if (!desc_ok(cache) || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    const int32_t row = cache->head_dim * elem_bytes(cache);
    int vec = 16;
    while (vec > 2 && (row % vec || !aligned(k, vec) || !aligned(v, vec) ||
                       !aligned(k_cache, vec) || !aligned(v_cache, vec)))
        vec >>= 1;
    if (row % vec || !aligned(k, vec) || !aligned(v, vec) || !aligned(k_cache, vec) ||
        !aligned(v_cache, vec) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int64_t total = (int64_t)num_tokens * 2 * cache->num_kv_heads * (row / vec);
    const int threads = 256;
    const int64_t sms = std::max(1, device_sm_count());
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads,
                                                                  sms * 16));
    const int64_t num_slots = (int64_t)cache->num_blocks * cache->block_size;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* kp = static_cast<const uint8_t*>(k);
    const uint8_t* vp = static_cast<const uint8_t*>(v);
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    cudaError_t err;
    switch (vec) {
        case 16:
            err = launch_pdl(write_kv_kernel<16>, dim3((unsigned)blocks), dim3(threads), 0, st,
                             kp, vp, slot_mapping, (int64_t)num_tokens, kc, vc,
                             cache->num_kv_heads, cache->block_size, num_slots, row);
            break;
        case 8:
            err = launch_pdl(write_kv_kernel<8>, dim3((unsigned)blocks), dim3(threads), 0, st,
                             kp, vp, slot_mapping, (int64_t)num_tokens, kc, vc,
                             cache->num_kv_heads, cache->block_size, num_slots, row);
            break;
        case 4:
            err = launch_pdl(write_kv_kernel<4>, dim3((unsigned)blocks), dim3(threads), 0, st,
                             kp, vp, slot_mapping, (int64_t)num_tokens, kc, vc,
                             cache->num_kv_heads, cache->block_size, num_slots, row);
            break;
        default:
            err = launch_pdl(write_kv_kernel<2>, dim3((unsigned)blocks), dim3(threads), 0, st,
                             kp, vp, slot_mapping, (int64_t)num_tokens, kc, vc,
                             cache->num_kv_heads, cache->block_size, num_slots, row);
            break;
    }
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int32_t pa_decode_path(int32_t num_q_heads, const pa_cache_desc* cache) {
    if (!desc_ok(cache) || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return -1;
    return fast_shape(cache, num_q_heads / cache->num_kv_heads) ? 1 : 0;
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
    const int32_t path = pa_decode_path(num_q_heads, cache);
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
    if (!fast && part > generic_max_partition(cache, group)) return PA_ERR_UNSUPPORTED;
    if (!aligned(q, elem_bytes(cache)) || !aligned(out, elem_bytes(cache)) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    const int32_t max_parts = num_parts(max_seq_len, part);
    if (max_parts > 65535) return PA_ERR_UNSUPPORTED;
    const size_t need = workspace_bytes(num_seqs, num_q_heads, max_seq_len, part, cache);
    if (need > 0 && (!workspace || workspace_bytes_given < need || !aligned(workspace, 256)))
        return PA_ERR_WORKSPACE;

    DecodeArgs a;
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

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    dim3 grid(max_parts, cache->num_kv_heads, num_seqs);
    cudaError_t err;
    if (fast) {
        CUtensorMap mk, mv;
        if (!cached_map(&mk, k_cache, cache, 0) || !cached_map(&mv, v_cache, cache, 1))
            return PA_ERR_CUDA;
        err = dispatch_fast(grid, mk, mv, a, st);
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
    if (max_parts > 1) {
        const unsigned mblocks = (unsigned)((int64_t)num_seqs * num_q_heads);
        const cudaError_t merr =
            cache->dtype == PA_F32
                ? launch_pdl(merge_kernel<float>, dim3(mblocks), dim3(kMergeThreads), 0, st, a)
                : launch_pdl(merge_kernel<__nv_bfloat16>, dim3(mblocks), dim3(kMergeThreads), 0,
                             st, a);
        if (merr != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
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
// up once per device with cudaGetSymbolAddress and cached.

static __device__ __align__(256) unsigned char g_no_alloc_workspace[PA_NO_ALLOC_WORKSPACE_BYTES];

namespace pa {
namespace {

void* g_no_alloc_ptr[kMaxDevices] = {nullptr};
std::mutex g_no_alloc_mutex;

// Device address of the static workspace for the current device, or nullptr
// if the lookup failed.  Runs cudaGetSymbolAddress on the first use per device.
void* no_alloc_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_no_alloc_mutex);
    if (g_no_alloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_workspace) != cudaSuccess) return nullptr;
        g_no_alloc_ptr[dev] = p;
    }
    return g_no_alloc_ptr[dev];
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
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, max_seq_len,
                                                  partition_tokens, cache);
    if (need > PA_NO_ALLOC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
    void* ws = pa::no_alloc_workspace();
    if (ws == nullptr) return PA_ERR_CUDA;
    return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     max_seq_len, num_q_heads, scale, partition_tokens, out, ws,
                     PA_NO_ALLOC_WORKSPACE_BYTES, cache, stream);
}
