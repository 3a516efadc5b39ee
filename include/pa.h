/*
 * libpa -- paged KV-cache decode attention for GB300 (sm_103a), C ABI.
 *
 * The KV cache of every running sequence is cut into fixed blocks of 16
 * tokens that need not be contiguous in memory; a per-sequence block table
 * maps logical block j to a physical block id, the way a page table maps
 * virtual pages to frames.  Sources:
 *   [P3] "vLLM Nedir? PagedAttention ile Production LLM Serving",
 *        sections "PagedAttention", "Bir istek motorun icinde",
 *        "Asil sisen sey agirlik degil, KV cache";
 *   [P4] "vLLM ve Triton ile maliyet optimizasyonu -- pratik karsilastirma",
 *        section 03 ("Yontem"), steps 1-3, copy-on-write and the paragraph
 *        on scaled dot-product attention;
 *   [P1] "Yerel LLM sistemlerinde backpressure ve olcekleme", section
 *        "KV butcesi" (grouped-query attention: 64 query heads, 8 KV heads).
 *
 * Conventions for every call:
 *   - Every function returns a pa_status (0 = PA_OK).  No exception or abort
 *     crosses the ABI.  After an error, pa_last_error_string() describes it
 *     (per calling thread).
 *   - The caller owns every device buffer, including the decode workspace
 *     (sized by pa_decode_workspace_bytes).  The library owns only the host
 *     allocator objects it creates.
 *   - Device calls take a CUDA stream as `void* stream` (a cudaStream_t;
 *     NULL = the legacy default stream), enqueue their kernels on it and
 *     return without synchronising.  Pointers named d_* are device memory;
 *     all others are host memory.
 *   - Physical cache layout, per K and per V:
 *       cache[num_blocks][num_kv_heads][16][head_dim]  (16-bit elements),
 *     so one (block, KV head) tile of 16 x head_dim elements is contiguous.
 *   - Element types: PA_F16 (IEEE binary16) or PA_BF16 (bfloat16) for q,
 *     k, v, the caches and the output.  head_dim 64 or 128.  The number of
 *     query heads per KV head (G = num_q_heads / num_kv_heads) is 1, 2, 4
 *     or 8; query head i reads KV head i / G.
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
    PA_ERR_INVALID = 1,      /* bad argument, shape, id or size */
    PA_ERR_OOM = 2,          /* the allocator's free queue cannot cover the request */
    PA_ERR_UNSUPPORTED = 3,  /* dtype / head_dim / group size with no compiled kernel */
    PA_ERR_SHARED_WRITE = 4, /* pa_seq_append_slots: a write would land in a block held by
                                several sequences and the call gave no room to report
                                the copy-on-write pair that must precede it */
    PA_ERR_CUDA = 5,         /* a CUDA call failed (launch, tensor map, copy) */
    PA_ERR_DEVICE = 6        /* a kernel flagged bad data (see pa_decode_check) */
} pa_status;

enum { PA_F16 = 0, PA_BF16 = 1 };
enum { PA_BLOCK_SIZE = 16 };

/* Device error bits reported by pa_decode_check. */
enum {
    PA_DEVERR_SEQ_LEN = 1,   /* a seq_len < 0 or > max_seq_len: clamped into range */
    PA_DEVERR_BLOCK_ID = 2,  /* a block id outside [0, num_blocks): read as zeros */
    PA_DEVERR_TIMEOUT = 4,   /* an internal wait gave up; the output is not valid */
    PA_DEVERR_GROUP = 8,     /* pa_decode_grouped: a group's offsets or shared prefix were
                                invalid; those sequences were decoded without sharing */
    PA_DEVERR_PLAN = 16      /* PA_DECODE_REUSE_PLAN: the workspace's plan did not fit this
                                call (records outside its buffers were skipped, or a length
                                differed from seq_lens); the output is not valid */
};

const char* pa_last_error_string(void);
const char* pa_version(void);

/* ------------------------------------------------------------------------
 * Host block allocator.  [P3] "PagedAttention" and "Bir istek motorun
 * icinde" steps 2 (allocate_slots) and 5 (finished blocks go back to the
 * free queue); [P4] section 03 step 3 (a block is taken only when the
 * current one is full) and the copy-on-write paragraph; [P3] last
 * paragraph of "PagedAttention" (shared blocks carry a reference count).
 *
 * Free queue: first in, first out.  Its initial order is `free_order` (a
 * permutation of 0..num_blocks-1) or 0,1,2,... when NULL; freed blocks join
 * the back in table order.  Sequence ids are 0,1,2,... and never reused.
 * An allocator object is not thread-safe; use one per thread or lock.
 * ---------------------------------------------------------------------- */
typedef struct pa_alloc pa_alloc_t;

typedef struct {
    int64_t num_blocks;
    int64_t free_blocks;    /* in the free queue */
    int64_t used_blocks;    /* reference count > 0 */
    int64_t shared_blocks;  /* reference count > 1 */
    int64_t refs;           /* sum of reference counts = table entries of live sequences */
    int64_t seqs;           /* live sequences */
    int64_t frag_tokens;    /* sum over live sequences of unfilled slots in their tables */
} pa_stats_t;

/* block_size must be 16.  *out receives the new allocator. */
int pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                    pa_alloc_t** out);
void pa_alloc_destroy(pa_alloc_t* a);

/* New empty sequence. */
int pa_seq_create(pa_alloc_t* a, int64_t* seq_id_out);

/* New sequence sharing the blocks that hold the parent's first
 * prefix_tokens tokens (0 <= prefix_tokens <= parent length); their
 * reference counts go up.  If the last shared block is only partly covered,
 * the first later write into it, by either holder, copies it (see
 * pa_seq_append_slots). */
int pa_seq_fork(pa_alloc_t* a, int64_t parent, int32_t prefix_tokens, int64_t* child_out);

/* Drop a sequence: every block's count goes down; a block reaching 0 joins
 * the free queue.  An unknown or already freed id is PA_ERR_INVALID. */
int pa_seq_free(pa_alloc_t* a, int64_t seq_id);

/* Reserve tokens_each new token slots for each of n_seqs distinct
 * sequences, sequence by sequence.  Slot of a token = physical block id * 16
 * + position % 16; a block is popped from the free queue when the position
 * starts a new block.  Writing into a block held by several sequences first
 * moves the writer onto a fresh block: the pair (source, destination) is
 * reported so the caller copies the block's contents on the device before
 * writing (cow_* arrays, capacity cow_capacity; *n_cow_out = pairs).
 *
 *   slot_mapping_out [n_seqs * tokens_each]  int64, sequence-major
 *   block_table_io   [n_seqs][max_blocks]    optional (NULL): row i is
 *                    updated in place with the entries that changed
 *   seq_lens_io      [n_seqs]                optional (NULL): new lengths
 *
 * All or nothing, and nothing changes when the call fails:
 *   PA_ERR_INVALID       unknown or repeated sequence, or a row would need
 *                        more than max_blocks entries;
 *   PA_ERR_SHARED_WRITE  a token would be written into a block another
 *                        sequence still holds and the copy-on-write pairs do
 *                        not fit cow_capacity (or the cow arrays are NULL):
 *                        the write would change the other holders' tokens;
 *   PA_ERR_OOM           the free queue cannot cover the new blocks plus the
 *                        copy targets.
 * The checks run in that order. */
int pa_seq_append_slots(pa_alloc_t* a, const int64_t* seq_ids, int32_t n_seqs,
                        int32_t tokens_each, int64_t* slot_mapping_out,
                        int32_t* cow_src_out, int32_t* cow_dst_out, int32_t cow_capacity,
                        int32_t* n_cow_out, int32_t* block_table_io, int32_t max_blocks,
                        int32_t* seq_lens_io);

/* Block table rows [n][max_blocks] (padding -1) and lengths of n sequences. */
int pa_seq_block_table(pa_alloc_t* a, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                       int32_t* table_out, int32_t* seq_lens_out);

int pa_alloc_stats(pa_alloc_t* a, pa_stats_t* out);

/* ------------------------------------------------------------------------
 * Cache write.  [P3] "Bir istek motorun icinde" step 2; [P4] section 03
 * steps 1-3: the new token's key and value rows go to the slot the
 * allocator handed out.
 *
 *   d_k, d_v          [num_tokens][num_kv_heads][head_dim]
 *   d_slot_mapping    [num_tokens] int64; slot s -> block s/16, row s%16.
 *                     s < 0 is padding and writes nothing; a slot whose
 *                     block is >= num_blocks writes nothing either.
 *   d_k_cache, d_v_cache  [num_blocks][num_kv_heads][16][head_dim]
 *
 * Bit copy: the cached bytes equal the input bytes.  Two tokens with the
 * same slot leave one of them (unspecified).  num_tokens == 0 is a no-op.
 * ---------------------------------------------------------------------- */
int pa_cache_write(const void* d_k, const void* d_v, const int64_t* d_slot_mapping,
                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                   void* d_k_cache, void* d_v_cache, int64_t num_blocks, int32_t dtype,
                   void* stream);

/* ------------------------------------------------------------------------
 * Copy-on-write block copy.  [P4] section 03: a block shared by several
 * sequences is kept once and copied when one holder writes into it; the
 * allocator reports the (source, destination) pairs in pa_seq_append_slots.
 *
 * For each pair i, block d_dst[i] becomes a copy of block d_src[i]: every KV
 * head's 16 rows, in K and in V (bit copy).  d_src, d_dst: [n_pairs] int32,
 * device.  A pair naming a block outside [0, num_blocks) is skipped.
 * Destinations must be distinct and must not be the source of another pair
 * in the same call (true of the allocator's pairs: destinations come fresh
 * from the free queue); otherwise the result is unspecified.  Enqueue it
 * before the cache write that caused the copy.
 * ---------------------------------------------------------------------- */
int pa_copy_blocks(void* d_k_cache, void* d_v_cache, int64_t num_blocks, int32_t num_kv_heads,
                   int32_t head_dim, const int32_t* d_src, const int32_t* d_dst, int32_t n_pairs,
                   void* stream);

/* ------------------------------------------------------------------------
 * Decode attention.  [P4] section 03: the maths of scaled dot-product
 * attention does not change under paging, only where K and V are read
 * from; the kernel follows the block table to gather them.  For every
 * sequence b and query head i (KV head h = i / G):
 *
 *   out[b][i] = sum_t softmax_t(scale * q[b][i] . K_b[t]) * V_b[t],
 *   t = 0 .. seq_lens[b]-1, K_b[t] = k_cache[table[b][t/16]][h][t%16].
 *
 *   d_q              [num_seqs][num_q_heads][head_dim]
 *   d_k_cache, d_v_cache  as for pa_cache_write (num_blocks blocks)
 *   d_block_tables   [num_seqs][max_blocks_per_seq] int32; entries past a
 *                    sequence's last block are never read
 *   d_seq_lens       [num_seqs] int32, the new token included
 *   max_seq_len      host-side bound on every seq_lens[b]; <= 0 means
 *                    max_blocks_per_seq * 16.  It sizes the workspace.
 *   d_out            [num_seqs][num_q_heads][head_dim]; seq_len 0 gives 0
 *   d_workspace      >= pa_decode_workspace_bytes(...) bytes, 256-byte
 *                    aligned, owned by the caller; its contents need no
 *                    initialisation and are overwritten by every call, so
 *                    calls sharing one workspace must not overlap in time.
 *
 * Built shapes: dtype PA_F16 or PA_BF16, head_dim 64 or 128, G =
 * num_q_heads / num_kv_heads of 1, 2, 4 or 8 (query heads h*G .. h*G+G-1
 * share KV head h); anything else returns PA_ERR_UNSUPPORTED.
 *
 * Accumulation is fp32 (online softmax over 16-token blocks; sequences
 * longer than one partition are split into partitions of 512, 1024 or 2048
 * tokens -- the prep kernel takes the largest that still leaves every SM
 * enough work -- whose partial results a second kernel merges), with one
 * rounding to the element type at the end.  Bad device data never faults:
 * it is clamped or read as zeros and flagged in the workspace
 * (pa_decode_check). */
size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_seq_len);

int pa_decode(const void* d_q, const void* d_k_cache, const void* d_v_cache, int64_t num_blocks,
              const int32_t* d_block_tables, int32_t max_blocks_per_seq,
              const int32_t* d_seq_lens, int32_t num_seqs, int32_t max_seq_len,
              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
              int32_t dtype, void* d_out, void* d_workspace, size_t workspace_bytes,
              void* stream);

/* Options for pa_decode_ex.  Zero-initialised = the pa_decode behaviour. */
enum {
    /* Reuse the plan the previous decode on this workspace computed (its
     * partition list and merge records): the prep kernel is skipped.  The
     * caller guarantees that seq_lens, num_seqs, max_seq_len, the head
     * counts, head_dim and (for pa_decode_grouped) the groups are those of
     * that call, and that it runs on this stream or one ordered after it;
     * q, the caches, block_tables' entries and out may differ -- e.g. the
     * layers of one decode step.  Not for pa_prefill.
     *   Checked on the host: the library records, per device and workspace
     *   address, the shapes (num_seqs, max_blocks_per_seq, max_seq_len, head
     *   counts, head_dim, number of groups) of the last planning call; a
     *   reuse without a matching record returns PA_ERR_INVALID and launches
     *   nothing.  A prefill on the workspace drops its record.
     *   Checked on the device: plan records that do not fit this call's
     *   workspace and sequences are skipped, and a planned length that
     *   differs from seq_lens is flagged; both set PA_DEVERR_PLAN.  Stale
     *   plan data therefore never addresses memory outside the call's
     *   buffers. */
    PA_DECODE_REUSE_PLAN = 1
};

typedef struct {
    int32_t variant;         /* 0 auto, 1 CUDA-core FMA + warp shuffles, 2 tensor-core
                                mma.sync, 3 tcgen05 with tensor-memory accumulators
                                (pa_prefill at head_dim 128 only) */
    int32_t flags;           /* PA_DECODE_* bits (decode calls only) */
    void* event_before_main; /* optional cudaEvent_t recorded just before the attention */
    void* event_after_main;  /* kernel and just after it, on the same stream */
    int32_t partition_tokens; /* decode calls: 0 = the prep kernel chooses (the default);
                                512, 1024 or 2048 = split every sequence into partitions of
                                exactly this many tokens (a sequence no longer than one
                                partition is then not split at all); anything else is
                                PA_ERR_INVALID.  Ignored with PA_DECODE_REUSE_PLAN (the
                                plan keeps its size).  The result is the same up to the
                                fp32 summation order, which the tests use to compare split
                                and unsplit decodes of one sequence. */
    int32_t reserved32;
    int64_t reserved[3];
} pa_decode_opts;

int pa_decode_ex(const void* d_q, const void* d_k_cache, const void* d_v_cache,
                 int64_t num_blocks, const int32_t* d_block_tables, int32_t max_blocks_per_seq,
                 const int32_t* d_seq_lens, int32_t num_seqs, int32_t max_seq_len,
                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                 int32_t dtype, void* d_out, void* d_workspace, size_t workspace_bytes,
                 void* stream, const pa_decode_opts* opts);

/* ------------------------------------------------------------------------
 * Decode with shared prefixes ("cascade").  [P3] "PagedAttention" last
 * paragraph and [P4] section 03: requests with a common prefix (a shared
 * system prompt, beam search, parallel sampling) point at the same physical
 * blocks.  Same result as pa_decode; the shared blocks are read from HBM
 * once per (group, KV head) instead of once per sequence, and their
 * attention is computed for all members at once on the tensor cores.
 *
 *   d_group_offsets       [num_groups + 1] int32, device: group g is the
 *                         contiguous sequences [off[g], off[g+1]);
 *                         off[0] = 0, off[num_groups] = num_seqs, non-decreasing
 *   d_group_prefix_tokens [num_groups] int32, device: tokens every member of g
 *                         holds in the same physical blocks as the group's
 *                         first member (a multiple of 16, at most any member's
 *                         length; 0 = no sharing).  The caller vouches that
 *                         the members' tables agree on those blocks (the
 *                         allocator's forks guarantee it).
 *   workspace             >= pa_decode_grouped_workspace_bytes(...)
 *
 * opts: as for pa_decode_ex (NULL = defaults); the events bracket the
 * attention kernel over the members' own tokens, not the prefix kernel.
 *
 * Invalid offsets or prefixes are flagged (PA_DEVERR_GROUP) and the affected
 * sequences are decoded without sharing -- still the correct result. */
size_t pa_decode_grouped_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                         int32_t max_seq_len);

int pa_decode_grouped(const void* d_q, const void* d_k_cache, const void* d_v_cache,
                      int64_t num_blocks, const int32_t* d_block_tables, int32_t max_blocks_per_seq,
                      const int32_t* d_seq_lens, int32_t num_seqs, int32_t max_seq_len,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                      int32_t dtype, const int32_t* d_group_offsets,
                      const int32_t* d_group_prefix_tokens, int32_t num_groups, void* d_out,
                      void* d_workspace, size_t workspace_bytes, void* stream,
                      const pa_decode_opts* opts);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) KV cache: half the bytes per token of a 16-bit cache, at some
 * accuracy risk.  [P1] section "1. KV cache tuketimi ve GPU bellek
 * tasmasi", the FP8 KV cache paragraph.  head_dim 128 only.
 *
 * Layout (bytes): K cache [num_blocks][num_kv_heads][16][128] as for 16-bit
 * caches; V cache dimension-major [num_blocks][num_kv_heads][128][16] (the
 * 16 tokens of one dimension are contiguous).  Scales: d_k_scale, d_v_scale
 * [num_kv_heads] float, device; a stored byte is
 * E4M3(fp32(x) * fp32(1 / scale[h])) -- rounded to nearest even, saturated to
 * +-448 -- and stands for byte * scale[h].
 *
 * pa_cache_write_fp8 quantises and scatters new tokens exactly like
 * pa_cache_write (k, v 16-bit of `dtype`).  pa_decode_fp8 is pa_decode over
 * the dequantised caches: q and out are 16-bit of `dtype`, q is rounded to
 * fp16 for the tensor cores (|q| must stay below 65504), accumulation fp32;
 * workspace as for pa_decode (pa_decode_workspace_bytes).  opts may be NULL;
 * its events work as for pa_decode_ex, variant must be 0 or 2 (the FP8 path
 * has only the tensor-core math; 1 gives PA_ERR_UNSUPPORTED). */
int pa_cache_write_fp8(const void* d_k, const void* d_v, const int64_t* d_slot_mapping,
                       int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                       const float* d_k_scale, const float* d_v_scale, void* d_k_cache8,
                       void* d_v_cache8, int64_t num_blocks, int32_t dtype, void* stream);

int pa_decode_fp8(const void* d_q, const void* d_k_cache8, const void* d_v_cache8,
                  const float* d_k_scale, const float* d_v_scale, int64_t num_blocks,
                  const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
                  int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                  int32_t head_dim, float scale, int32_t dtype, void* d_out, void* d_workspace,
                  size_t workspace_bytes, void* stream, const pa_decode_opts* opts);

/* ------------------------------------------------------------------------
 * Multi-query paged attention: chunked prefill with decode tokens in the
 * same call.  "Yerel LLM sistemlerinde backpressure ve olcekleme", section
 * "4. Prefill ve decode", and "vLLM Nedir? PagedAttention ile Production LLM
 * Serving", section "Chunked prefill": a long prompt is cut into pieces that
 * fit a step's token budget and each iteration computes one piece together
 * with the running sequences' decode tokens; the piece's K/V fill the
 * sequence's blocks over several steps.
 *
 * Sequence b holds seq_lens[b] tokens in its blocks after the piece's K/V
 * were written (pa_cache_write); its piece is the last
 * Q_b = q_offsets[b+1] - q_offsets[b] of them (a decode token is a piece of
 * one).  Query j of the piece sits at position seq_lens[b] - Q_b + j and
 * attends causally to tokens 0 .. seq_lens[b] - Q_b + j:
 *   out[t, i] = softmax_j(scale * q[t, i] . K[j, i / G]) V[j, i / G].
 *
 *   d_q, d_out     [num_q_tokens][num_q_heads][head_dim] 16-bit, the pieces
 *                  back to back (16-byte aligned)
 *   d_q_offsets    [num_seqs + 1] int32, device: q_offsets[0] = 0,
 *                  non-decreasing, q_offsets[num_seqs] = num_q_tokens
 *   caches, d_block_tables, d_seq_lens, max_seq_len, scale, dtype: as for
 *                  pa_decode (max_seq_len bounds every seq_lens[b])
 *   d_workspace    >= pa_prefill_workspace_bytes(...) bytes, 256-byte
 *                  aligned, caller-owned; calls sharing it must not overlap
 *   opts           NULL, or events recorded around the attention kernel;
 *                  variant 0 = tcgen05 at head_dim 128 and mma.sync at 64,
 *                  2 = mma.sync, 3 = tcgen05 (head_dim 128)
 *
 * fp32 accumulation, one rounding to dtype.  Bad device data never faults: a
 * length outside [0, max_seq_len], a piece longer than its sequence or
 * offsets out of order are flagged (PA_DEVERR_SEQ_LEN) and clamped, block
 * ids outside the pool read as zeros (PA_DEVERR_BLOCK_ID); the error bits
 * are read with pa_decode_check on this workspace.
 *
 * Resources: the tcgen05 kernel runs one CTA per SM with ~226 KB of shared
 * memory and allocates all 512 tensor-memory columns of its SM for the
 * CTA's lifetime (the allocation waits while another kernel on the SM
 * holds tensor memory); num_blocks * num_kv_heads * 16 must stay below
 * 2^31 (tensor-map row coordinates). */
size_t pa_prefill_workspace_bytes(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                  int32_t num_kv_heads);

int pa_prefill(const void* d_q, const void* d_k_cache, const void* d_v_cache, int64_t num_blocks,
               const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
               const int32_t* d_q_offsets, int32_t num_seqs, int32_t num_q_tokens,
               int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
               float scale, int32_t dtype, void* d_out, void* d_workspace, size_t workspace_bytes,
               void* stream, const pa_decode_opts* opts);

/* Waits for `stream`, then reads the device error bits the last decode (or
 * prefill) using this workspace left (PA_DEVERR_*; 0 = clean) into
 * *error_bits.  Returns PA_ERR_DEVICE when any bit is set. */
int pa_decode_check(const void* d_workspace, void* stream, int32_t* error_bits);

/* ------------------------------------------------------------------------
 * Diagnostic with no counterpart on the pages: the bounded wait that every
 * kernel of this library uses on its mbarriers, shown to end.  One CTA waits
 * on a barrier nothing arrives at; after limit_ns (0 < limit_ns <= 1e9) the
 * wait gives up and the kernel returns normally, writing to d_status[0..3]
 * (int32, device): whether the wait succeeded (0 expected), the error bits
 * (PA_DEVERR_TIMEOUT expected), the CTA's abort flag (1 expected) and the
 * microseconds waited.  Asynchronous on `stream`. */
int pa_selftest_bounded_wait(int64_t limit_ns, int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * Decode without any allocation.  The pages have no counterpart: this is a
 * convenience for callers that cannot allocate device memory or pass a
 * workspace (a fixed, pre-planned memory budget, a plugin or callback that
 * owns no device memory, code that must not allocate next to a caching
 * allocator).  Same arguments and result as pa_decode, minus the workspace:
 * the scratch is one static 64 MiB device array per device, held from the
 * library's module load until process exit.
 *   - Batches whose pa_decode_workspace_bytes(num_seqs, num_q_heads,
 *     head_dim, max_seq_len) exceeds 64 MiB are rejected with
 *     PA_ERR_INVALID (nothing is launched).
 *   - Calls no cudaMalloc/cudaFree or other allocating routine.
 *   - The first call on a device looks up the array's device address (and
 *     may load the module); make that first call before any stream capture.
 *     The address is kept for the process: after cudaDeviceReset the
 *     array may move, so do not call this entry point again on a device
 *     that was reset.
 *   - Every call on a device shares the array and leaves its contents
 *     behind; each call rewrites what it reads, but calls whose kernels may
 *     overlap on the GPU (unordered streams) race on it and must not be
 *     issued.  Device error bits of the last call are not readable through
 *     this entry point.
 * ---------------------------------------------------------------------- */
int pa_decode_noalloc(const void* d_q, const void* d_k_cache, const void* d_v_cache,
                      int64_t num_blocks, const int32_t* d_block_tables, int32_t max_blocks_per_seq,
                      const int32_t* d_seq_lens, int32_t num_seqs, int32_t max_seq_len,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                      int32_t dtype, void* d_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
