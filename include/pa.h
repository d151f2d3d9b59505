/*
 * pa.h -- C ABI of the PagedAttention decode library (libpa.so, sm_103a).
 *
 * The problem, as the pages state it:
 *  - "LLM Serving Engine Shootout: vLLM vs TensorRT-LLM vs SGLang vs
 *    llama.cpp", 3.1 PagedAttention Mechanics: each sequence's KV cache lives
 *    in fixed-size physical blocks (16 or 32 tokens) of one pool; a block table
 *    maps logical block index to physical block; the logit of the query against
 *    key j is q . k_j / sqrt(d_head), with k_j fetched through
 *    BlockTable[floor(j / block_size)].
 *  - zhichai.net (Chinese original), section 1 diagram: tokens 0-15 of a
 *    sequence in physical block #7, tokens 16-31 in physical block #2; token j
 *    sits at row j mod block_size of its block.
 *  - "Serving engines" (inference.tusharamrit.in), How vLLM works: given a
 *    block table and a slot mapping, the kernel gathers the right K/V vectors
 *    from scattered memory; blocks may be shared by several sequences
 *    (copy-on-write), and a write forks only the block being written.
 *
 * Conventions for every call:
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; the caller owns all memory.  No call allocates
 *    device memory or keeps state between calls, except a per-device error
 *    word (see pa_device_errors) and the fixed scratch array that
 *    pa_decode_static_workspace uses.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every compute call only validates its arguments on the host,
 *    enqueues kernels on `stream` and returns; results are ready when the
 *    stream reaches that point.
 *  - Layouts (row-major, element type given by `dtype`, 2 bytes each; the
 *    caches of the *_fp8 calls hold one-byte codes, see "FP8 KV cache"):
 *      k_cache, v_cache  [num_blocks, num_kv_heads, block_size, head_dim]
 *      query, out        [num_seqs, num_q_heads, head_dim]
 *      block_tables      int32 [num_seqs, max_blocks_per_seq]; entry
 *                        (i, b) is the physical block of logical block b of
 *                        sequence i; entries past a sequence's last block are
 *                        never read (-1 by convention)
 *      context_lens      int32 [num_seqs]; tokens 0..context_lens[i]-1 of
 *                        sequence i are attended to (the newest token included)
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads) (contiguous
 *    query-head groups).
 *  - Errors: host-side checks happen before any launch and return
 *    PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED with nothing enqueued.  A failed
 *    launch returns PA_ERR_CUDA.  Data errors that only the device can see
 *    (a block-table entry outside [0, num_blocks), a slot outside the pool, a
 *    context length beyond the table or beyond max_context_len, a wait that
 *    ran out of time) never trap: the kernel skips the bad access (masking
 *    the tokens it would have read, or skipping the bad row), records a bit
 *    in the device error word, and the caller reads it with
 *    pa_device_errors.  No call aborts or throws.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, too-small workspace */
    PA_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels are built for */
    PA_ERR_CUDA = 3           /* a CUDA runtime call or launch failed */
} pa_status;

typedef enum pa_dtype {
    PA_FP16 = 0,              /* IEEE binary16 */
    PA_BF16 = 1               /* bfloat16 */
} pa_dtype;

/* Bits of the device error word (see pa_device_errors). */
#define PA_DEVERR_BAD_BLOCK 1u   /* a needed block-table entry was outside [0, num_blocks) */
#define PA_DEVERR_BAD_SLOT  2u   /* a slot_mapping entry was >= num_blocks * block_size */
#define PA_DEVERR_BAD_LEN   4u   /* a context length was < 0, > max_blocks_per_seq * block_size
                                    or > max_context_len */
#define PA_DEVERR_TIMEOUT   8u   /* a wait for staged KV data ran past its time limit */
#define PA_DEVERR_WORKSPACE 16u  /* a split-context join counter in the workspace did not
                                    start at zero (see pa_decode_workspace_size) */
#define PA_DEVERR_PREFIX    32u  /* pa_decode_shared_prefix(_fp8): the groups do not cover the batch,
                                    a group is larger than max_group_size, members of a group
                                    give different prefix lengths, or a member's table names
                                    other blocks than the group's for its shared prefix */

/*
 * pa_reshape_and_cache -- write each new token's key and value into its slot
 * of the paged cache ("Serving engines", How vLLM works: slot mapping).
 *
 *   for every t < num_tokens with s = slot_mapping[t] >= 0, every h:
 *     k_cache[s / block_size, h, s % block_size, :] = key[t, h, :]
 *     v_cache[s / block_size, h, s % block_size, :] = value[t, h, :]
 *
 * key, value       device, [num_tokens, num_kv_heads, head_dim]; row t starts
 *                  at element t * key_stride (value_stride); heads are
 *                  contiguous inside a row.  Strides in elements, >=
 *                  num_kv_heads * head_dim and a multiple of 8.
 * k_cache, v_cache device, updated in place; every other slot is untouched.
 * slot_mapping     device int64 [num_tokens]; negative = skip the token.
 * The copy is bit-exact.  Slots must be distinct within one call (two tokens
 * writing one slot leave either value).  A slot >= num_blocks * block_size is
 * skipped and sets PA_DEVERR_BAD_SLOT.
 * Pointers 16-byte aligned.  head_dim in {64, 128}, block_size in {16, 32}.
 */
pa_status pa_reshape_and_cache(const void *key, const void *value,
                               int64_t key_stride, int64_t value_stride,
                               void *k_cache, void *v_cache,
                               const int64_t *slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t num_blocks,
                               int32_t dtype, void *stream);

/*
 * Number of partitions pa_decode uses: 1 when partition_size == 0 or
 * max_context_len <= partition_size, else ceil(max_context_len / partition_size).
 */
int32_t pa_decode_num_partitions(int32_t max_context_len, int32_t partition_size);

/*
 * Bytes of workspace pa_decode needs (0 when it runs as one partition).
 * Layout, P = pa_decode_num_partitions(...), R = num_seqs * num_q_heads,
 * each array starting at a 256-byte aligned offset, in this order:
 *   counters  uint32 [PA_DECODE_COUNTER_BYTES / 4]  join counters (below)
 *   m  float [R, P]      max over the partition of scale * q.k_j * log2(e)
 *   l  float [R, P]      sum over the partition of 2^(scale*q.k_j*log2(e) - m)
 *   o  float [R, P, head_dim]  the partition's normalised attention output
 * Row r = seq * num_q_heads + head.  A sequence's partitions
 * p < ceil(ctx / partition_size) are written, except that when the join runs
 * inside the decode kernel (P <= 32 and num_seqs * num_kv_heads <= 65536) a
 * sequence with a single partition writes its output directly and no partial.
 *
 * Join counters: word seq * num_kv_heads + kv_head counts the partitions of
 * that sequence and KV head that have finished; the last one joins them and
 * sets the word back to zero.  The counter words must therefore be ZERO the
 * first time a workspace is used (cudaMemset the first PA_DECODE_COUNTER_BYTES
 * once after allocating it); every completed pa_decode call leaves them zero
 * again, for any later shape, since the counters never move and no partial is
 * ever stored over them.  A counter that is found not to have started at zero
 * sets PA_DEVERR_WORKSPACE and that row's output is not written.
 */
#define PA_DECODE_COUNTER_BYTES (256u * 1024u)

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                int32_t max_context_len, int32_t partition_size);

/*
 * pa_decode -- single-query paged attention for a batch of sequences
 * ("LLM Serving Engine Shootout", 3.1 PagedAttention Mechanics).
 *
 *   out[i, h, :] = sum_j softmax_j(scale * q[i, h, :] . K_j) V_j,
 *   j < context_lens[i], K_j = k_cache[block_tables[i, j / bs], h / G, j % bs, :]
 *   (V_j alike), G = num_q_heads / num_kv_heads.  context_lens[i] == 0 gives 0.
 *
 * Softmax and accumulation are fp32 (online softmax in one pass over the
 * tokens); out is rounded to dtype (round to nearest even).
 * partition_size == 0, or max_context_len <= partition_size: one pass per
 * (sequence, KV head) writes out directly; workspace may be NULL.
 * partition_size > 0 (a multiple of 16): the tokens of each sequence are cut
 * into partitions of partition_size, each partition is attended to
 * separately into `workspace` (layout above, counter words zero), and the
 * partitions are joined by log-sum-exp: inside the decode kernel, by the last
 * partition of each (sequence, KV head) to finish, when there are at most 32
 * partitions; otherwise by pa_decode_reduce on the same stream.
 * max_context_len must be >= every context_lens[i] (sizes the launch).
 * Pointers (out, query, caches) 16-byte aligned; head_dim in {64, 128};
 * block_size in {16, 32}; num_q_heads / num_kv_heads in 1..8.
 * The caches are read-only here; out must not overlap any input.
 */
pa_status pa_decode(void *out, const void *query,
                    const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens,
                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t block_size, int64_t num_blocks,
                    float scale, int32_t max_context_len, int32_t partition_size,
                    void *workspace, size_t workspace_bytes,
                    int32_t dtype, void *stream);

/*
 * pa_decode_reduce -- join split-context partitions by log-sum-exp:
 *   M = max_p m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p
 * over the ceil(context_lens[i] / partition_size) partitions of each row
 * (0 partitions: out = 0).  `workspace` holds the partials in the layout of
 * pa_decode_workspace_size for the same num_seqs, num_q_heads, head_dim,
 * max_context_len and partition_size (partition_size > 0); the counter words
 * are not read.  pa_decode calls this itself when it splits into more
 * partitions than its kernel joins; it is exported so partials from elsewhere
 * can be joined.
 */
pa_status pa_decode_reduce(void *out, const void *workspace, const int32_t *context_lens,
                           int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                           int32_t max_context_len, int32_t partition_size,
                           int32_t dtype, void *stream);

/*
 * pa_decode_shared_prefix -- pa_decode for a batch whose sequences come in
 * groups that share a prefix held in the same physical blocks (copy-on-write
 * sharing: "LLM Serving Engine Shootout", 3.2 Copy-on-Write and 4
 * RadixAttention; "Serving engines", How vLLM works).  The result is
 * pa_decode's for the same arguments (the same formula, within rounding);
 * the difference is the memory traffic: the K/V of a group's shared prefix
 * is read once per group (per 128 query heads of it) instead of once per
 * sequence.
 *
 * group_start   device int32 [num_groups + 1]: group g is the sequences
 *               group_start[g] .. group_start[g+1]-1; group_start[0] = 0,
 *               non-decreasing, group_start[num_groups] = num_seqs (every
 *               sequence in exactly one group; a sequence that shares nothing
 *               is a group of its own).
 * prefix_lens   device int32 [num_seqs]: the number of leading tokens of
 *               sequence i whose blocks are the same physical blocks for
 *               every member of its group (equal within a group; 0 = none).
 *               Only whole partitions of it are shared: member i takes
 *               partitions p < min(prefix_lens[i] / partition_size,
 *               ceil(context_lens[i] / partition_size) - 1) from the shared
 *               pass and the rest from the per-sequence decode.
 * num_groups    1 .. num_seqs;  max_group_size >= every group's size (sizes
 *               the launch).
 * partition_size  > 0, a multiple of 16, at most 8192; with one partition
 *               (max_context_len <= partition_size) nothing can be shared and
 *               the call is pa_decode.
 * Other arguments, the workspace (pa_decode_workspace_size bytes, counter
 * words zero) and the accuracy are as for pa_decode; dtype fp16 or bf16
 * caches (FP8 caches: pa_decode_shared_prefix_fp8 below).  Input errors only
 * the device can see set PA_DEVERR_PREFIX (see above): the output of the
 * sequences concerned is then unspecified, never a fault.
 */
pa_status pa_decode_shared_prefix(void *out, const void *query,
                                  const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens,
                                  const int32_t *group_start, const int32_t *prefix_lens,
                                  int32_t num_groups, int32_t max_group_size,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                  float scale, int32_t max_context_len, int32_t partition_size,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t dtype, void *stream);

/*
 * pa_prefill -- chunked-prefill attention over the paged cache ("Serving
 * engines", How vLLM works: chunked prefill slices a long prompt into pieces;
 * "LLM Serving Engine Shootout", 1: prefill attends over all prompt tokens).
 *
 * Sequence i appends q_len_i = query_start[i+1] - query_start[i] tokens, query
 * rows query_start[i] .. query_start[i+1]-1, whose K/V are already in the
 * cache (pa_reshape_and_cache of those tokens), so the sequence now holds
 * context_lens[i] >= q_len_i tokens.  Chunk row t sits at position
 * p = context_lens[i] - q_len_i + t and attends causally:
 *   out[row, h, :] = sum_{j <= p} softmax_j(scale q[row, h] . K_j) V_j
 * with K_j, V_j read through the block table as in pa_decode.
 *
 * query, out     device, [total_q, num_q_heads, head_dim], dtype; 16-byte aligned
 * query_start    device int32 [num_seqs + 1], non-decreasing, query_start[0] = 0
 * max_q_len      >= every q_len_i (sizes the launch)
 * Softmax and accumulation fp32; out rounded to dtype.  scale > 0.  head_dim
 * in {64, 128}, block_size in {16, 32}, num_q_heads / num_kv_heads in 1..8
 * (every shape runs on the tcgen05 kernel: two 128-row query tiles per CTA
 * when max_q_len * G > 128, one otherwise).  A
 * q_len_i larger than context_lens[i] or than max_q_len, or a context longer
 * than the table, skips that sequence and sets PA_DEVERR_BAD_LEN.  A block id
 * outside [0, num_blocks) for a token in use sets PA_DEVERR_BAD_BLOCK; that
 * block is never read and its tokens are left out of the softmax.
 */
pa_status pa_prefill(void *out, const void *query, const int32_t *query_start,
                     const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                     const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int64_t num_blocks, float scale,
                     int32_t dtype, void *stream);

/*
 * FP8 KV cache.  The cache stores one byte per element, an FP8 E4M3 code
 * (1 sign, 4 exponent bits with bias 7, 3 fraction bits, no infinities,
 * largest magnitude 448), with one scale per cache: code e stands for
 * k_scale * e (K) or v_scale * e (V).  This halves the KV bytes the decode
 * reads (zhichai.net section 4 counts FP8 at 1 byte per element; "Serving
 * engines" lists KV quantisation among the shared engine features).
 * Layout [num_blocks, num_kv_heads, block_size, head_dim] as above, uint8.
 */

/*
 * pa_reshape_and_cache_fp8 -- pa_reshape_and_cache into FP8 caches: every
 * element x of the new rows (src_dtype fp16 or bf16) is stored as the E4M3
 * code of x / scale, the quotient an IEEE single-precision division, rounded
 * to the nearest code (ties to even), magnitudes beyond 448 clamped to 448.
 * k_scale, v_scale finite and > 0.  Other arguments as pa_reshape_and_cache.
 */
pa_status pa_reshape_and_cache_fp8(const void *key, const void *value,
                                   int64_t key_stride, int64_t value_stride,
                                   void *k_cache, void *v_cache,
                                   const int64_t *slot_mapping,
                                   int32_t num_tokens, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                   int32_t src_dtype, float k_scale, float v_scale,
                                   void *stream);

/*
 * pa_decode_fp8 -- pa_decode over FP8 caches: K_j = k_scale * e4m3(k code),
 * V_j = v_scale * e4m3(v code).  Codes are converted exactly to fp16 in the
 * kernel and both products run in fp16 with fp32 accumulation; k_scale joins
 * the softmax scale and v_scale multiplies the output.  query/out fp16
 * (dtype = PA_FP16) or bf16 (PA_BF16): bf16 queries are scaled by a power of
 * two per (sequence, KV head) so that their largest magnitude fits fp16, then
 * rounded to fp16 (exact for every value down to 2^-31 of the largest), and
 * the power of two is taken back out of the softmax scale.  head_dim 64 or 128,
 * block_size 16 or 32.  Workspace as for pa_decode.
 */
pa_status pa_decode_fp8(void *out, const void *query,
                        const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                        const int32_t *context_lens,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int64_t num_blocks,
                        float scale, float k_scale, float v_scale,
                        int32_t max_context_len, int32_t partition_size,
                        void *workspace, size_t workspace_bytes,
                        int32_t dtype, void *stream);

/*
 * pa_prefill_fp8 -- pa_prefill over FP8 caches, K_j and V_j as in
 * pa_decode_fp8.  The tcgen05 kernel copies each step's codes into shared
 * memory and widens them there to fp16 (exact), so both products run in fp16
 * with fp32 accumulation; k_scale joins the softmax scale and v_scale
 * multiplies the output.  bf16 queries (dtype = PA_BF16) are scaled by a
 * power of two per row (token, head) so that the row's largest magnitude
 * fits fp16, rounded to fp16 (exact for every value down to 2^-31 of the
 * largest), and the power of two is taken back out of that row's softmax
 * scale; out is written in dtype.  k_scale, v_scale finite and > 0.  Other
 * arguments, shapes and error behaviour as pa_prefill.
 */
pa_status pa_prefill_fp8(void *out, const void *query, const int32_t *query_start,
                         const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                         const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, float scale,
                         float k_scale, float v_scale, int32_t dtype, void *stream);

/*
 * pa_decode_shared_prefix_fp8 -- pa_decode_shared_prefix over FP8 caches: the
 * result is pa_decode_fp8's for the same arguments (K_j, V_j, scales and
 * queries as there); the shared pass reads the codes of a group's shared
 * prefix once per group (per 128 query heads of it) and widens them as
 * pa_prefill_fp8 does.  Group arguments, workspace and device checks as
 * pa_decode_shared_prefix.
 */
pa_status pa_decode_shared_prefix_fp8(void *out, const void *query,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens,
                                      const int32_t *group_start, const int32_t *prefix_lens,
                                      int32_t num_groups, int32_t max_group_size,
                                      int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int64_t num_blocks, float scale,
                                      float k_scale, float v_scale,
                                      int32_t max_context_len, int32_t partition_size,
                                      void *workspace, size_t workspace_bytes,
                                      int32_t dtype, void *stream);

/*
 * pa_copy_blocks -- copy-on-write fork of whole physical blocks ("Serving
 * engines", How vLLM works: sequences share physical blocks until one writes;
 * the write forks only the block being written).
 *
 *   for every k < num_pairs, with (s, d) = (block_mapping[2k], block_mapping[2k+1]):
 *     k_cache[d, :, :, :] = k_cache[s, :, :, :];  v_cache[d] = v_cache[s]
 *
 * k_cache, v_cache  device, [num_blocks, num_kv_heads, block_size, head_dim],
 *                   16-byte aligned; updated in place, bit-exact.
 * block_mapping     device int64 [num_pairs, 2].  Destinations must be
 *                   distinct and none may also be a source in the same call
 *                   (otherwise the result is undefined).  A pair with an id
 *                   outside [0, num_blocks) is skipped and sets
 *                   PA_DEVERR_BAD_BLOCK.
 * head_dim in {64, 128}, block_size in {16, 32}.  16-bit caches (fp16 or
 * bf16, 2 bytes per element); pa_copy_blocks_fp8 is the same over FP8 caches
 * (1 byte per element).
 */
pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                         int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, void *stream);
pa_status pa_copy_blocks_fp8(void *k_cache, void *v_cache, const int64_t *block_mapping,
                             int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int64_t num_blocks, void *stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools, typically the device
 * pool and a pinned host pool ("Serving engines", How vLLM works: a preempted
 * sequence's blocks are swapped out to host memory and back in later).
 *
 *   for every k < num_pairs: dst block block_mapping[2k+1] = src block block_mapping[2k]
 *
 * src, dst       each device memory, managed memory, or pinned host memory
 *                (cudaHostAlloc / cudaHostRegister; the library reaches it
 *                through its device-mapped address); pageable host memory is
 *                refused with PA_ERR_INVALID_ARG.  Both 16-byte aligned; pool
 *                i has blocks of block_bytes (a multiple of 16) laid out
 *                back to back.  Call once for the K pool and once for V.
 * block_mapping  int64 [num_pairs, 2] in device or pinned host memory;
 *                destinations distinct; ids outside [0, src_num_blocks) or
 *                [0, dst_num_blocks) skip the pair and set PA_DEVERR_BAD_BLOCK.
 * The copy is one kernel on `stream`, bit-exact.  As with every call, host
 * memory must stay valid until the stream has passed this point.
 */
pa_status pa_swap_blocks(const void *src, void *dst, const int64_t *block_mapping,
                         int32_t num_pairs, int64_t block_bytes, int64_t src_num_blocks,
                         int64_t dst_num_blocks, void *stream);

/*
 * pa_decode_static_workspace -- pa_decode for callers that cannot allocate
 * device memory.  The pages have no counterpart to this call.  Some callers
 * of a decode kernel may not call cudaMalloc at all: a serving framework that
 * has reserved nearly all device memory for its own KV pool and hands none of
 * it to libraries, a plugin running under a host runtime that owns every
 * allocation on the device, or a real-time enqueue path that cannot risk the
 * device-wide synchronisation an allocation may cause.
 *
 * Same arguments and result as pa_decode, without workspace / workspace_bytes:
 * the split-context partials and join counters go to a fixed array of
 * PA_STATIC_WORKSPACE_BYTES inside the library (a __device__ variable, so
 * every device that loads the library holds that much memory until the
 * process exits).  The call allocates nothing and calls no allocating routine.
 *  - Arguments are checked as pa_decode checks them, with the same statuses;
 *    then a shape whose pa_decode_workspace_size exceeds
 *    PA_STATIC_WORKSPACE_BYTES is rejected with PA_ERR_UNSUPPORTED.  Nothing
 *    is enqueued in either case.
 *  - The first call on a device looks up that device's copy of the array
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents.  Each call that splits clears the join counters it uses
 *    (cudaMemsetAsync on `stream`, no allocation) before its kernels; nothing
 *    else needs to start at zero.  Calls whose kernels overlap on the GPU
 *    (different streams, or different host threads, without ordering between
 *    them) race on the array: order them.
 */
#define PA_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)

pa_status pa_decode_static_workspace(void *out, const void *query,
                                     const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *context_lens,
                                     int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     float scale, int32_t max_context_len, int32_t partition_size,
                                     int32_t dtype, void *stream);

/*
 * Read and clear the device error word of the current device after waiting
 * for `stream` to finish.  *flags receives the PA_DEVERR_* bits raised since
 * the last call (by any call on any stream of this device).  Returns PA_OK or
 * PA_ERR_CUDA.
 */
pa_status pa_device_errors(void *stream, uint32_t *flags);

/*
 * Self-test of the device-side wait limit (no counterpart on the pages; it
 * exists so the failure path of every staged-data wait can be exercised
 * without a fault).  Launches one CTA on `stream` that waits on a barrier
 * nothing ever completes; the wait gives up after its limit (about 1 s),
 * sets PA_DEVERR_TIMEOUT in the device error word and the CTA exits, leaving
 * the context usable.  Returns after the launch: PA_OK or PA_ERR_CUDA.
 */
pa_status pa_selftest_bounded_wait(void *stream);

/* Static description of a status code (never NULL). */
const char *pa_status_string(int32_t status);

/* Library ABI version: 4 (2 added the join counters to the workspace, 3
   pa_decode_shared_prefix, 4 the FP8 forms of pa_prefill,
   pa_decode_shared_prefix and pa_copy_blocks). */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
