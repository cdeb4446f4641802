/*
 * pa.h -- C ABI of the paged-attention decode library (libpa.so).
 *
 * Two operations, both asynchronous on the caller's CUDA stream and both
 * reading and writing only caller-owned device memory:
 *
 *   pa_write_kv  scatter each new token's K and V rows into its cache slot
 *                ("vLLM PagedAttention: from memory fragmentation to slot
 *                mapping", §6: the backend writes new K/V to physical slots
 *                named by the slot mapping; paper notes' block lifecycle table:
 *                decode fills the next slot of the last block);
 *   pa_decode    single-query multi-head / grouped-query attention whose K/V
 *                history is read through a block table (same page §3-§4:
 *                logical block floor(t/B), offset t mod B, slot =
 *                table[logical]*B + offset; "vLLM source walkthrough:
 *                PagedAttention and Continuous Batching" §1.8: per-block walk,
 *                V2 partitions merged by a reduce step; "PagedAttention"
 *                glossary: the result equals attention over contiguous K/V).
 *
 * Cache layout (both caches, one layer): [num_blocks][num_kv_heads][block_size]
 * [head_dim], head_dim contiguous.  One (block, kv head) tile is block_size *
 * head_dim contiguous elements.  This is the glossary page's teaching layout,
 * not vLLM's split-x K layout.
 *
 * Element types: PA_F32 (IEEE binary32) or PA_BF16 (bfloat16).  q, k, v, out
 * and both caches share the cache's type; accumulation is fp32.
 *
 * Ownership: the caller allocates and frees every buffer (caches, tables,
 * lengths, q, out, workspace).  The library allocates no device memory and
 * keeps no per-call state; it caches one TMA descriptor pair per host thread.
 *
 * Memory: caches and workspaces must be device (or managed) memory.  The
 * per-call arguments marked "device or pinned" below -- queries, new K/V,
 * slots, tables, lengths, query starts and outputs -- may instead be
 * page-locked host memory: the kernels then read or write it directly over
 * the host link (NVLink-C2C on Grace-Blackwell), with no staging copy.
 * Pageable host memory, or a cache or workspace outside device memory, is
 * refused with PA_ERR_INVALID_ARG (PA_ERR_WORKSPACE for the workspace)
 * before anything is launched.
 *
 * Errors: argument problems found on the host return a status and launch
 * nothing.  Problems only visible on the device (a needed block-table entry
 * outside [0, num_blocks), a sequence longer than its table or than
 * max_seq_len, a slot outside the cache, a pipeline wait that exceeded its
 * bound) never fault: the kernel skips the offending access, sets a bit in a
 * device error word and carries on; read it with pa_last_device_error().
 * No C++ exception crosses this interface.
 *
 * Debugging: with PA_DEBUG=1 in the environment (read at every call), each
 * call first synchronises its stream, copies its index arrays to the host and
 * checks them as a whole.  Duplicate slots, two copies into one block (or,
 * inside one pool, onto a source), entries or slots outside the pool, lengths
 * past their bounds, query rows out of order and appends into a block that
 * another table also reaches are then refused with
 * PA_ERR_INVALID_ARG before launch (the first violation is printed to
 * stderr).  This is slow and is not for use under stream capture.
 *
 * Tracing: each call is an NVTX range of its own name (pa_write_kv,
 * pa_decode, ...) around its checks and launches.
 *
 * CUDA graphs: the launching calls can be captured on a stream and replayed.
 * A replay reads whatever the captured buffers hold at that time.  The grid
 * is fixed at capture from the host bounds (max_seq_len, max_q_len, token
 * and pair counts), so only the buffers' contents may change between
 * replays, with lengths staying within those bounds.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes */
    PA_ERR_UNSUPPORTED = 2,   /* valid request this build cannot run */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    PA_ERR_CUDA = 4           /* a CUDA call or launch failed */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Geometry of one layer's K and V caches (both have this shape). */
typedef struct {
    int32_t num_blocks;    /* physical blocks in the pool                */
    int32_t block_size;    /* B: tokens per block                        */
    int32_t num_kv_heads;  /* Hkv                                        */
    int32_t head_dim;      /* D                                          */
    int32_t dtype;         /* pa_dtype                                   */
} pa_cache_desc;

/* Device error bits reported by pa_last_device_error(). */
#define PA_DEVERR_TABLE_ENTRY 1u  /* a needed table entry was outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN     2u  /* seq_lens[i] > max_seq_len or > max_blocks*B     */
#define PA_DEVERR_SLOT        4u  /* a slot was >= num_blocks * block_size            */
#define PA_DEVERR_TIMEOUT     8u  /* a pipeline wait gave up after its bound          */
#define PA_DEVERR_BLOCK_PAIR 16u  /* a copy pair named a block outside its cache       */
#define PA_DEVERR_GROUP      32u  /* a shared-prefix group, member or length out of range */

/*
 * pa_write_kv -- cache write through slot_mapping.
 *
 * k, v          device or pinned, [num_tokens][num_kv_heads][head_dim], cache dtype.
 * slot_mapping  device or pinned int64 [num_tokens]; token j goes to slot s =
 *               slot_mapping[j]: block s / B, row s % B, for every kv head.
 *               s < 0 means "skip this token".  Slots must be distinct within
 *               one call (two writers of one slot race).
 * k_cache, v_cache  device caches, written in place.
 * stream        cudaStream_t (NULL = legacy default stream).
 * The copy is bit-exact.  num_tokens == 0 is a no-op.  Writing into a block
 * that several sequences share is the caller's error (copy it first).
 */
pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache,
                      const pa_cache_desc* cache, void* stream);

/*
 * pa_write_kv_positions -- the same cache write, with each token's slot
 * computed on the device from its sequence and position through the block
 * table ("vLLM PagedAttention: from memory fragmentation to slot mapping" §6:
 * positions and the device block table give the slot mapping; §3: slot =
 * table[pos / B] * B + pos % B).
 *
 * seq_ids, positions  device or pinned int32 [num_tokens]; token j belongs to sequence
 *               seq_ids[j] at position positions[j].  A negative id or
 *               position means "skip"; an id >= num_seqs, a position past the
 *               table, or a table entry outside [0, num_blocks) is skipped and
 *               reported (PA_DEVERR_TABLE_ENTRY).
 * block_tables  device or pinned int32 [num_seqs][max_blocks_per_seq].
 * Other arguments as pa_write_kv.
 */
pa_status pa_write_kv_positions(const void* k, const void* v, const int32_t* seq_ids,
                                const int32_t* positions, int32_t num_tokens,
                                const int32_t* block_tables, int32_t num_seqs,
                                int32_t max_blocks_per_seq, void* k_cache, void* v_cache,
                                const pa_cache_desc* cache, void* stream);

/*
 * pa_copy_blocks -- whole-block copies for copy-on-write and swapping
 * (PagedAttention engineering notes, nxmr.cn, §4.2: before a shared, partly
 * filled block is written, take a new block and copy the old block's K/V into
 * it; paper notes on swapping: a preempted sequence's blocks move to CPU
 * memory and back).
 *
 * src_k, src_v  source caches, src_num_blocks blocks of the geometry `cache`
 *               describes (its num_blocks field is not used here).
 * dst_k, dst_v  destination caches, dst_num_blocks blocks; may be the source
 *               caches themselves (copy-on-write inside one pool).
 * block_pairs   int64 [num_pairs][2] of (src block, dst block), copied as if in
 *               order; a destination must not appear twice nor be a source in
 *               the same call (those copies race).  Pairs outside either pool
 *               are skipped and reported (PA_DEVERR_BLOCK_PAIR).
 * Every pointer may be device memory or page-locked host memory (a swap pool
 * allocated with cudaHostAlloc or registered with cudaHostRegister); pageable
 * host memory is refused with PA_ERR_INVALID_ARG.  Bit-exact.
 */
pa_status pa_copy_blocks(const void* src_k, const void* src_v, int32_t src_num_blocks,
                         void* dst_k, void* dst_v, int32_t dst_num_blocks,
                         const int64_t* block_pairs, int32_t num_pairs,
                         const pa_cache_desc* cache, void* stream);

/*
 * Partition size (tokens, a multiple of block_size) that pa_decode uses when
 * called with partition_tokens == 0.  Depends only on the arguments and on
 * the current device's SM count.  Returns <= 0 on invalid arguments.
 */
int32_t pa_decode_partition_tokens(int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_seq_len, const pa_cache_desc* cache);

/*
 * Workspace bytes pa_decode needs for these arguments (0 when no sequence can
 * span more than one partition).  partition_tokens == 0 selects the automatic
 * size.  Layout, P = ceil(max_seq_len / partition_tokens):
 *   float acc[num_seqs][num_q_heads][P][head_dim]   unnormalised sum_t w_t v_t
 *   float ml [num_seqs][num_q_heads][P][2]          (m, l)
 * with s_t = scale * q.k_t, m = log2(e) * max_t s_t (base-2 units),
 * w_t = exp(s_t - max_t s_t), l = sum_t w_t, all over the partition's tokens.
 * Cells of sequences that fit one partition are not written.
 */
size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                 int32_t max_seq_len, int32_t partition_tokens,
                                 const pa_cache_desc* cache);

/*
 * pa_decode -- out[i][h] = sum_{t < T_i} softmax_t(scale * q[i][h].k_t) v_t,
 * with k_t, v_t the cache rows of kv head floor(h / (Hq/Hkv)) at slot
 * table[i][t / B] * B + t % B, and T_i = seq_lens[i].  T_i == 0 gives a zero
 * row.
 *
 * q              device or pinned [num_seqs][num_q_heads][head_dim], cache dtype.
 * block_tables   device or pinned int32 [num_seqs][max_blocks_per_seq]; entries at or
 *                beyond ceil(T_i / B) are never read (pad with -1).
 * seq_lens       device or pinned int32 [num_seqs].
 * max_seq_len    host upper bound of seq_lens (sizes the grid; no device
 *                read-back).  Must satisfy max_seq_len <= max_blocks_per_seq*B.
 * scale          softmax scale (1/sqrt(head_dim) for standard attention).
 * partition_tokens  split-K partition (multiple of B), or 0 for automatic.
 *                Sequences longer than one partition are computed per
 *                partition and merged with a log-sum-exp reduction.
 * out            device or pinned [num_seqs][num_q_heads][head_dim], cache dtype,
 *                round-to-nearest-even from fp32.
 * workspace      device, >= pa_decode_workspace_bytes(...) bytes, 256-byte
 *                aligned; may be NULL when that size is 0.
 * The result is bitwise reproducible for fixed arguments on a fixed device.
 */
pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_q_heads, float scale, int32_t partition_tokens,
                    void* out, void* workspace, size_t workspace_bytes,
                    const pa_cache_desc* cache, void* stream);

/*
 * pa_decode_append -- one decode step in one call: each sequence's newest
 * token is written to the caches, then pa_decode runs over the same
 * arguments.  Sequence i's newest token is position T_i - 1 (T_i =
 * seq_lens[i] counts it; "PagedAttention" glossary, upstream and downstream:
 * decode appends one slot per step; "PagedAttention engineering notes"
 * (nxmr.cn) §3.1: each generated token's K/V goes to the next slot of the
 * sequence's current block), and its rows k_new[i], v_new[i] go to slot
 * table[i][(T_i - 1) / B] * B + (T_i - 1) % B of both caches.  The caches and
 * the output are bit for bit those of pa_write_kv_positions(k_new, v_new,
 * seq_ids = 0 .. num_seqs - 1, positions = T_i - 1) followed by pa_decode.
 *
 * On the TMA decode kernel (pa_decode_path 1, head_dim up to 128, k_new and
 * v_new 16-byte aligned) the write is fused into the decode: the CTA whose partition holds
 * position T_i - 1 attends to the new rows in place of the slot's old
 * contents and stores them, so the step is one launch shorter.  Otherwise
 * the cache write (slots from the lengths and tables) runs first, then the
 * decode.
 *
 * k_new, v_new   device or pinned [num_seqs][num_kv_heads][head_dim], cache dtype.
 * k_cache, v_cache  written at the appended slots.
 * T_i == 0 appends nothing.  A length outside [0, min(max_seq_len,
 * max_blocks_per_seq * B)] or a bad table entry at the appended position
 * appends nothing and is reported (PA_DEVERR_SEQ_LEN, PA_DEVERR_TABLE_ENTRY),
 * as pa_decode reports it.  The appended slot must belong to this sequence
 * alone (a block shared with another table is copied first: pa_copy_blocks);
 * two sequences appending to one slot is undefined.  Both are refused under
 * PA_DEBUG.
 * Other arguments, the workspace and the errors as pa_decode.
 */
pa_status pa_decode_append(const void* q, const void* k_new, const void* v_new,
                           void* k_cache, void* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads,
                           float scale, int32_t partition_tokens, void* out,
                           void* workspace, size_t workspace_bytes,
                           const pa_cache_desc* cache, void* stream);

/*
 * pa_decode_shared_prefix -- pa_decode for a batch in which groups of
 * sequences share their leading blocks: a common prompt prefix held once and
 * referenced by several block tables ("vLLM source walkthrough: PagedAttention
 * and Continuous Batching" §1.6: blocks with ref_cnt > 1 shared by sequences
 * with a common prefix; "PagedAttention engineering notes" (nxmr.cn) §4.1:
 * forked sequences point at the same prompt blocks; "vLLM PagedAttention:
 * from memory fragmentation to slot mapping" §5).  The result is pa_decode's
 * over the same tables, within the same tolerance: one softmax over every
 * visible key, now taken as the log-sum-exp merge of the shared blocks'
 * partials with each member's own ("Efficient Memory Management for LLM
 * Serving with PagedAttention" paper notes, blockwise softmax example).  What
 * changes is the reads: the shared blocks are read once per kv head and tile
 * of (member, query head) rows (16 rows, 8 for groups of up to 8 query heads
 * per kv head) instead of once per member.
 *
 * Group k (0 <= k < num_groups) has the member sequences
 * members[member_start[k] .. member_start[k+1]), each sequence in at most
 * one group.  Its members' first prefix_blocks[k] table entries name the same
 * physical blocks (the caller's promise, checked under PA_DEBUG).  A member
 * may be shorter than the shared blocks: it sees only its own T_i keys.
 *
 * seq_group      device or pinned int32 [num_seqs]: k for a member of group k,
 *                -1 (or any negative value) for a sequence in no group.  It must
 *                agree with the member lists: a sequence listed in a group but
 *                not marked here, or the reverse, gets an undefined output
 *                (refused under PA_DEBUG).
 * member_start   device or pinned int32 [num_groups + 1], from 0, non-decreasing.
 * members        device or pinned int32 [member_start[num_groups]], sequence ids.
 * prefix_blocks  device or pinned int32 [num_groups], each in [0, max_prefix_blocks].
 * max_group_size    host bound of the groups' sizes (sizes the grid).
 * max_prefix_blocks host bound of prefix_blocks, <= max_blocks_per_seq.
 * workspace      device, >= pa_decode_shared_prefix_workspace_bytes(...) bytes,
 *                256-byte aligned (never NULL when num_groups > 0 on the TMA
 *                kernel's shapes: every member is merged).
 * mode           PA_SHARED_ONCE: read the shared blocks once per row tile;
 *                PA_SHARED_PLAIN: run the plain pa_decode over the same tables;
 *                PA_SHARED_AUTO: once when a row tile holds m >= 2 members
 *                (m = 8 rows, 16 for groups of more than 8 query heads per kv
 *                head, over that group size) and max_prefix_blocks * B *
 *                (1 - 1/m) >= 1024 tokens, plain otherwise.  The plain decode
 *                reads each member's shared blocks, mostly from L2; reading
 *                them once costs an extra merge per member, which pays only
 *                when enough reads are saved (measured: a 512-token prefix at
 *                4 query heads per kv head is 1.5% faster plain, a 4096-token
 *                one 16% faster once; one member per tile is 13% faster plain).
 * Other arguments as pa_decode.  A group id, member id, member list (offsets
 * outside [0, member_start[num_groups]] or longer than max_group_size) or
 * shared-block count out of range on the device is skipped and reported
 * (PA_DEVERR_GROUP); the affected members' outputs are then undefined.
 * Shapes that pa_decode_path does not send to kernel 1, and num_groups == 0,
 * run the plain pa_decode over the same tables in every mode: same result.
 */
typedef enum { PA_SHARED_AUTO = 0, PA_SHARED_ONCE = 1, PA_SHARED_PLAIN = 2 } pa_shared_mode;

/* 1 when pa_decode_shared_prefix with these arguments reads the shared
 * blocks once per row tile, 0 when it runs the plain decode, < 0 for invalid
 * arguments. */
int32_t pa_decode_shared_prefix_mode(int32_t num_q_heads, int32_t max_prefix_blocks,
                                     int32_t mode, const pa_cache_desc* cache);
size_t pa_decode_shared_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                               int32_t max_seq_len, int32_t max_prefix_blocks,
                                               int32_t partition_tokens,
                                               const pa_cache_desc* cache);
pa_status pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs,
                                  int32_t max_seq_len, int32_t num_q_heads, float scale,
                                  int32_t partition_tokens, const int32_t* seq_group,
                                  const int32_t* member_start, const int32_t* members,
                                  const int32_t* prefix_blocks, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_blocks,
                                  int32_t mode, void* out, void* workspace,
                                  size_t workspace_bytes, const pa_cache_desc* cache,
                                  void* stream);

/*
 * pa_prefill -- multi-query (chunked prefill) paged attention with a causal
 * mask ("vLLM source walkthrough: PagedAttention and Continuous Batching"
 * §2.8: prefill rows and decode rows in one batch, long prompts in chunks;
 * "vLLM PagedAttention: from memory fragmentation to slot mapping" §6: query
 * start locations slice the packed tokens per request, positions set the
 * causal boundary).
 *
 * Sequence i owns the packed query rows [query_start_loc[i],
 * query_start_loc[i+1]): its last L_i positions (their K/V already written
 * to the cache).  Row r is at position p = T_i - L_i + (r - query_start_loc[i])
 * and attends to keys 0..p of its sequence:
 *   out[r][h] = sum_{t <= p} softmax_t(scale * q[r][h].k_t) v_t,
 * kv head floor(h / (Hq/Hkv)), keys read through the block table as in
 * pa_decode.  A decode row is a sequence with L_i = 1.
 *
 * q, out           device or pinned [total_q][num_q_heads][head_dim], cache dtype.
 * query_start_loc  device or pinned int32 [num_seqs + 1], non-decreasing, last = total_q.
 * max_q_len        host upper bound of L_i (sizes the grid).
 * Other arguments as pa_decode.  L_i > T_i is reported (PA_DEVERR_SEQ_LEN)
 * and that sequence's rows are left untouched.  bf16 with head_dim a multiple
 * of 16 up to 128 (16-48 in a 64-column tile, 80-112 in a 128-column tile,
 * whose extra columns are zero), block_size 8 or a multiple of 16, a group size of at most 128 and scale >= 0
 * runs on the TMA + tcgen05 kernel (tensor-memory accumulators); other valid
 * shapes (head_dim <= 256) and scales on a warp-level tensor-core kernel
 * (bf16, head_dim a multiple of 16, 16-byte aligned q and caches), else on
 * CUDA cores: a tiled kernel when the rows are whole 16-byte pieces and the
 * caches 16-byte aligned, else a generic one.  The tensor-core kernels take
 * the softmax weights into P V as two bf16 parts (the weight rounded, and its
 * rounding error rounded), about 16 significant bits.
 */
pa_status pa_prefill(const void* q, const int32_t* query_start_loc, int32_t total_q,
                     int32_t max_q_len, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                     int32_t num_q_heads, float scale, void* out, const pa_cache_desc* cache,
                     void* stream);

/*
 * Which decode kernel these arguments select: 1 = the TMA + tensor-core
 * kernel (bf16, head_dim a multiple of 16 up to 128, or 256 with groups of
 * two or more query heads per kv head, block_size 8 or a multiple
 * of 16 up to 256, any group size: a group of more than 16 query heads is
 * split into CTAs of 16 that read the same K/V tiles), 2 = the warp-level tensor-core
 * kernel (bf16, head_dim a multiple of 16 up to 128 that kernel 1 does not
 * take, groups of 5 or more query heads; used when q is 4-byte and the caches
 * 16-byte aligned), 0 = a CUDA-core kernel (any other valid shape, and every
 * fp32 cache: the tiled kernel when head_dim is at most 256 with rows of
 * whole 16-byte pieces and the caches are 16-byte aligned, else the generic
 * one), < 0 = invalid arguments.
 */
int32_t pa_decode_path(int32_t num_q_heads, const pa_cache_desc* cache);

/*
 * pa_decode_no_alloc -- pa_decode for callers that cannot allocate device
 * memory when they run attention (for example a plugin hook of an inference
 * engine that forbids allocation during execution, or a process working in a
 * fixed, pre-reserved memory budget).  The pages have no counterpart to it.
 *
 * Same arguments and result as pa_decode, minus the workspace: the split-K
 * workspace is a fixed array of PA_NO_ALLOC_WORKSPACE_BYTES (32 MiB) inside
 * the library, held by every GPU that loads libpa.so until the process exits.
 * The call allocates nothing itself.
 * - The first call on each device looks the array's device address up (with
 *   that device current) and caches it, with the id of the device's current
 *   context, for the life of the process; make that first call before any
 *   stream capture.  After a cudaDeviceReset the context, and with it the
 *   array's address, changes: the next call notices the new context and looks
 *   the address up again, so that call too must come before any capture.
 * - A request of more than 65535 partitions (the longest sequence over the
 *   partition size) returns PA_ERR_UNSUPPORTED, as pa_decode does.  A request
 *   whose workspace (pa_decode_workspace_bytes with the same arguments)
 *   exceeds PA_NO_ALLOC_WORKSPACE_BYTES returns PA_ERR_WORKSPACE.  Neither
 *   launches anything.
 * - All calls on a device share the one array, which keeps the last call's
 *   contents.  Nothing in it needs to start at zero: every cell the merge reads
 *   is written earlier in the same call.  Calls whose execution overlaps on the
 *   GPU (different streams without ordering between them) race on the array;
 *   order them on one stream or synchronise between them.
 */
#define PA_NO_ALLOC_WORKSPACE_BYTES (32u << 20)
pa_status pa_decode_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                             int32_t num_q_heads, float scale, int32_t partition_tokens,
                             void* out, const pa_cache_desc* cache, void* stream);

/*
 * pa_check_wait_timeout -- checks the bounded wait that every kernel here
 * uses between its roles (copy issue, MMA issue, softmax).  One CTA of
 * max(32, expected) threads initialises an mbarrier that needs `expected`
 * arrivals, makes `arrivals` of them, and waits for the phase with a bound of
 * `limit_cycles` SM clocks.
 * - arrivals == expected: the phase completes and nothing is raised.
 * - arrivals < expected: nothing completes the phase; the wait gives up after
 *   the bound, PA_DEVERR_TIMEOUT is raised and the kernel returns.  Nothing
 *   faults and the context stays usable.
 * Read the outcome with pa_last_device_error().  Needs 1 <= expected <= 1024,
 * 0 <= arrivals <= expected and 1000 <= limit_cycles <= 2^31, else
 * PA_ERR_INVALID_ARG.  Asynchronous on `stream`.
 */
pa_status pa_check_wait_timeout(int32_t expected, int32_t arrivals, int64_t limit_cycles,
                                void* stream);

/* Human-readable name of a status code (static string). */
const char* pa_status_str(pa_status status);

/* Synchronises the current device, returns the PA_DEVERR_* bits raised since
 * the last call, and clears them.  Returns -1 if the read itself failed. */
int32_t pa_last_device_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
