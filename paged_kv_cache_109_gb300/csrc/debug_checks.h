// debug_checks.h -- host-side validation of a call's index arguments, on when
// the environment has PA_DEBUG=1 (read at every call).
//
// The kernels already skip and report what they can see from one CTA (a
// table entry outside the pool, a slot past the pool, a length past its bound).
// This pass sees the whole call before anything is launched, so it also finds
// what no CTA can: two tokens written to one slot, or two copies into one
// block, which would race.  It synchronises the stream and copies the index
// arrays to the host, so it is for debugging only.  A failed check prints the
// first violation to stderr and the call returns PA_ERR_INVALID_ARG without
// launching.
//
// Ref counts are not the library's: a write into a block that sequences share
// is refused by the host block pool before the call.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "pa.h"

namespace pa {
namespace debug {

inline bool enabled() {
    const char* e = std::getenv("PA_DEBUG");
    return e && std::strcmp(e, "1") == 0;
}

// n elements of a device or page-locked host array, once the stream's earlier
// work (which may produce them) has finished.
template <typename T>
bool fetch(std::vector<T>& out, const T* p, size_t n, cudaStream_t st) {
    out.resize(n);
    if (n == 0) return true;
    if (cudaStreamSynchronize(st) != cudaSuccess) return false;
    return cudaMemcpy(out.data(), p, n * sizeof(T), cudaMemcpyDefault) == cudaSuccess;
}

inline pa_status fail(const char* what, long long a, long long b) {
    std::fprintf(stderr, "pa debug check: %s (%lld, %lld)\n", what, a, b);
    return PA_ERR_INVALID_ARG;
}

// Slots: each is < 0 (skipped) or below num_slots, and no slot appears twice.
inline pa_status check_slot_list(std::vector<int64_t> slots, int64_t num_slots) {
    for (size_t j = 0; j < slots.size(); ++j)
        if (slots[j] >= num_slots) return fail("slot past the pool (token, slot)", (long long)j, slots[j]);
    std::sort(slots.begin(), slots.end());
    for (size_t j = 1; j < slots.size(); ++j)
        if (slots[j] >= 0 && slots[j] == slots[j - 1])
            return fail("two tokens write one slot (slot, -)", slots[j], -1);
    return PA_OK;
}

inline pa_status check_slots(const int64_t* slot_mapping, int32_t n, int64_t num_slots,
                             cudaStream_t st) {
    std::vector<int64_t> s;
    if (!fetch(s, slot_mapping, (size_t)n, st)) return PA_ERR_CUDA;
    return check_slot_list(std::move(s), num_slots);
}

// Slots from (sequence, position) through the block tables, as the write
// kernel computes them; an entry the kernel would report is an error here.
inline pa_status check_positions(const int32_t* seq_ids, const int32_t* positions, int32_t n,
                                 const int32_t* tables, int32_t num_seqs, int32_t max_blocks,
                                 const pa_cache_desc* c, cudaStream_t st) {
    std::vector<int32_t> sid, pos, tab;
    if (!fetch(sid, seq_ids, (size_t)n, st) || !fetch(pos, positions, (size_t)n, st) ||
        !fetch(tab, tables, (size_t)num_seqs * max_blocks, st))
        return PA_ERR_CUDA;
    std::vector<int64_t> slots((size_t)n, -1);
    for (int32_t j = 0; j < n; ++j) {
        const int32_t s = sid[j], p = pos[j];
        if (s < 0 || p < 0) continue;
        if (s >= num_seqs || (int64_t)p >= (int64_t)max_blocks * c->block_size)
            return fail("sequence or position outside the tables (token, position)", j, p);
        const int32_t id = tab[(size_t)s * max_blocks + p / c->block_size];
        if (id < 0 || id >= c->num_blocks) return fail("table entry outside the pool (token, id)", j, id);
        slots[j] = (int64_t)id * c->block_size + p % c->block_size;
    }
    return check_slot_list(std::move(slots), (int64_t)c->num_blocks * c->block_size);
}

// Lengths within both bounds and every table entry that a length needs inside
// the pool; with query_start (prefill), rows ordered and L_i <= T_i.
inline pa_status check_tables(const int32_t* tables, int32_t max_blocks, const int32_t* seq_lens,
                              int32_t num_seqs, int32_t max_seq_len, const int32_t* query_start,
                              int32_t total_q, const pa_cache_desc* c, cudaStream_t st) {
    std::vector<int32_t> tab, len, qs;
    if (!fetch(tab, tables, (size_t)num_seqs * max_blocks, st) ||
        !fetch(len, seq_lens, (size_t)num_seqs, st) ||
        (query_start && !fetch(qs, query_start, (size_t)num_seqs + 1, st)))
        return PA_ERR_CUDA;
    const int32_t B = c->block_size;
    for (int32_t i = 0; i < num_seqs; ++i) {
        const int32_t T = len[i];
        if (T < 0 || T > max_seq_len || (int64_t)T > (int64_t)max_blocks * B)
            return fail("length outside its bounds (sequence, length)", i, T);
        for (int32_t b = 0; b < (T + B - 1) / B; ++b) {
            const int32_t id = tab[(size_t)i * max_blocks + b];
            if (id < 0 || id >= c->num_blocks)
                return fail("needed table entry outside the pool (sequence, id)", i, id);
        }
        if (query_start) {
            const int32_t L = qs[i + 1] - qs[i];
            if (qs[i] < 0 || L < 0 || qs[i + 1] > total_q)
                return fail("query rows out of order (sequence, start)", i, qs[i]);
            if (L > T) return fail("more query rows than positions (sequence, rows)", i, L);
        }
    }
    return PA_OK;
}

// A decode step's appends (pa_decode_append): each sequence with T > 0 writes
// position T - 1 of its own table.  Refused: two sequences on one slot, and
// a slot in a block that another sequence's table also reaches (a shared
// block must be copied before it is written).  The lengths and entries
// themselves are check_tables' business.
inline pa_status check_appends(const int32_t* tables, int32_t max_blocks, const int32_t* seq_lens,
                               int32_t num_seqs, const pa_cache_desc* c, cudaStream_t st) {
    std::vector<int32_t> tab, len;
    if (!fetch(tab, tables, (size_t)num_seqs * max_blocks, st) ||
        !fetch(len, seq_lens, (size_t)num_seqs, st))
        return PA_ERR_CUDA;
    const int32_t B = c->block_size;
    std::vector<int32_t> owners((size_t)c->num_blocks, 0);   // tables reaching each block
    for (int32_t i = 0; i < num_seqs; ++i)
        for (int32_t b = 0; b < (len[i] + B - 1) / B; ++b) {
            const int32_t id = tab[(size_t)i * max_blocks + b];
            if (id >= 0 && id < c->num_blocks) ++owners[id];
        }
    std::vector<int64_t> slots;
    for (int32_t i = 0; i < num_seqs; ++i) {
        if (len[i] <= 0) continue;
        const int32_t id = tab[(size_t)i * max_blocks + (len[i] - 1) / B];
        if (id < 0 || id >= c->num_blocks) continue;
        if (owners[id] > 1)
            return fail("append into a block another table reaches (sequence, block)", i, id);
        slots.push_back((int64_t)id * B + (len[i] - 1) % B);
    }
    return check_slot_list(std::move(slots), (int64_t)c->num_blocks * B);
}

// Shared-prefix groups: member lists ordered from 0, within the host bounds,
// every member a valid sequence in exactly one group whose seq_group entry
// names it (and -1 for the other sequences), and every member's first
// prefix_blocks table entries the same physical blocks as the group's first
// member's.
inline pa_status check_groups(const int32_t* tables, int32_t max_blocks, int32_t num_seqs,
                              const int32_t* seq_group, const int32_t* member_start,
                              const int32_t* members, const int32_t* prefix_blocks,
                              int32_t num_groups, int32_t max_group_size,
                              int32_t max_prefix_blocks, cudaStream_t st) {
    std::vector<int32_t> tab, sg, ms, mem, pb;
    if (!fetch(tab, tables, (size_t)num_seqs * max_blocks, st) ||
        !fetch(sg, seq_group, (size_t)num_seqs, st) ||
        !fetch(ms, member_start, (size_t)num_groups + 1, st) ||
        !fetch(pb, prefix_blocks, (size_t)num_groups, st))
        return PA_ERR_CUDA;
    if (ms[0] != 0) return fail("member_start[0] is not 0 (group, start)", 0, ms[0]);
    for (int32_t k = 0; k < num_groups; ++k) {
        const int32_t cnt = ms[k + 1] - ms[k];
        if (cnt < 0 || cnt > max_group_size)
            return fail("group size outside [0, max_group_size] (group, size)", k, cnt);
        if (pb[k] < 0 || pb[k] > max_prefix_blocks)
            return fail("shared blocks outside [0, max_prefix_blocks] (group, blocks)", k, pb[k]);
    }
    if (!fetch(mem, members, (size_t)ms[num_groups], st)) return PA_ERR_CUDA;
    std::vector<int32_t> owner((size_t)num_seqs, -1);
    for (int32_t k = 0; k < num_groups; ++k) {
        for (int32_t j = ms[k]; j < ms[k + 1]; ++j) {
            const int32_t i = mem[j];
            if (i < 0 || i >= num_seqs) return fail("member outside the batch (group, id)", k, i);
            if (owner[i] >= 0) return fail("sequence in two groups (sequence, group)", i, k);
            owner[i] = k;
            for (int32_t b = 0; b < pb[k]; ++b)
                if (tab[(size_t)i * max_blocks + b] != tab[(size_t)mem[ms[k]] * max_blocks + b])
                    return fail("member's leading block differs from the group's (sequence, block)",
                                i, b);
        }
    }
    for (int32_t i = 0; i < num_seqs; ++i)
        if (sg[i] != owner[i]) return fail("seq_group disagrees with the members (sequence, group)", i, sg[i]);
    return PA_OK;
}

// Copy pairs inside both pools; no block is written twice, and inside one pool
// no destination is also a source (the result would depend on the order).
inline pa_status check_pairs(const int64_t* pairs, int32_t n, int32_t src_blocks,
                             int32_t dst_blocks, bool same_pool, cudaStream_t st) {
    std::vector<int64_t> pr;
    if (!fetch(pr, pairs, (size_t)n * 2, st)) return PA_ERR_CUDA;
    std::vector<int64_t> dst, src;
    for (int32_t j = 0; j < n; ++j) {
        const int64_t s = pr[2 * (size_t)j], d = pr[2 * (size_t)j + 1];
        if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks)
            return fail("copy pair outside its pool (pair, src)", j, s);
        dst.push_back(d);
        src.push_back(s);
    }
    std::sort(dst.begin(), dst.end());
    for (size_t j = 1; j < dst.size(); ++j)
        if (dst[j] == dst[j - 1]) return fail("two copies into one block (block, -)", dst[j], -1);
    if (same_pool) {
        std::sort(src.begin(), src.end());
        for (int64_t d : dst)
            if (std::binary_search(src.begin(), src.end(), d))
                return fail("a destination is also a source (block, -)", d, -1);
    }
    return PA_OK;
}

}  // namespace debug
}  // namespace pa
