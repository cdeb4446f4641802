// prefill_args.cuh -- arguments and tuning knobs of the multi-query (chunked
// prefill) paged attention kernels.
//
// Sequence i owns the packed query rows [query_start[i], query_start[i+1]):
// its last L_i positions, row r at position p = T_i - L_i + (r - start),
// attending to keys 0..p ("vLLM source walkthrough: PagedAttention and
// Continuous Batching" §2.8: chunked prefill and decode rows in one batch;
// "vLLM PagedAttention: from memory fragmentation to slot mapping" §6: query
// start locations slice the tokens per request, positions set the causal
// boundary).
#pragma once

#include <cuda.h>

#include "decode_generic.cuh"
#include "ptx.cuh"

#ifndef PA_PREFILL_KEYS
#define PA_PREFILL_KEYS 128   // keys per block of the tcgen05 prefill (64 or 128)
#endif
#ifndef PA_PREFILL_PRODUCERS
#define PA_PREFILL_PRODUCERS 2   // warps issuing the tcgen05 prefill's K/V copies
#endif

namespace pa {

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
    int32_t tokens_per_tile;        // 128 / group (tensor-core kernel)
    float scale_log2;
};

}  // namespace pa
