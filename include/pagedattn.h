/*
 * pagedattn.h -- C ABI of the GB300 paged-KV decode library.
 *
 * What it computes.  Decode-time scaled dot-product attention of each
 * sequence's single new query against its key/value cache, where the cache is
 * stored as fixed 16-token physical blocks and a per-sequence block table maps
 * logical block i to a physical block ("vLLM: treating the KV cache as virtual
 * memory", section 破除误解: the formula is unchanged, only the layout; the
 * kernel follows the block table with one indirection per block).  Around it:
 * writing each step's new K/V rows into their paged slots, copying whole
 * blocks for copy-on-write, and a host-side block pool that produces the
 * tables.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every function returns an int status (pa_status).  On a non-zero status
 *   pa_last_error() returns a message for the calling thread.
 * - Device pointers are raw CUDA device addresses owned by the caller.  The
 *   library never allocates, frees or retains device memory, and keeps no
 *   pointer after a call returns.  Host pointers are read (or written) during
 *   the call only.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Device work is enqueued asynchronously on it; a PA_OK return means the
 *   work was validated and launched, not that it finished.
 * - Host-side validation (shapes, dtype, alignment, pointer presence) happens
 *   before any launch; a failing check launches nothing.
 * - Data-dependent checks (block ids, slots, context lengths read on the
 *   device) never fault: an out-of-range value is clamped or skipped and a
 *   device status word is set.  pa_check_status() reads and clears it.
 *   Every device-side wait is bounded; a wait that runs out sets
 *   PA_ERR_DEVICE_TIMEOUT in the same word instead of hanging.
 * - Element types: PA_F32, PA_F16, PA_BF16.  Caches, queries, new K/V and the
 *   output all share one dtype per call.  head_dim is 64 or 128.
 * - Shapes whose workspace would come near the range of size_t are refused
 *   (PA_ERR_INVALID_ARG) by every entry point and workspace-size query.
 * - Every compute entry point opens an NVTX range named after itself in the
 *   "pagedattn" domain, so an NVTX-aware profiler attributes each call and
 *   the kernels it launched; without a profiler attached this costs a test
 *   of an unset function pointer.
 *
 * Layouts (row-major, contiguous)
 * -------------------------------
 *   k_cache, v_cache : [num_blocks][num_kv_heads][16][head_dim]
 *                      (one (block, head) tile = 16 * head_dim elements,
 *                       contiguous; physical block p, token offset o of head h
 *                       is element ((p * num_kv_heads + h) * 16 + o) * head_dim)
 *   q, out           : [num_seqs][num_q_heads][head_dim]
 *   k, v (new rows)  : [num_tokens][num_kv_heads][head_dim]
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq]
 *   context_lens     : int32 [num_seqs]
 *   slot_mapping     : int64 [num_tokens], slot = physical_block * 16 + offset
 *   src_dst_pairs    : int64 [num_pairs][2]
 *
 * Query head h reads KV head h / (num_q_heads / num_kv_heads) (contiguous
 * groups; GQA when the ratio exceeds one).
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#define PA_BLOCK_SIZE 16

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,    /* bad shape, pointer, alignment or workspace size */
  PA_ERR_UNSUPPORTED = 2,    /* dtype, head_dim or head grouping not built */
  PA_ERR_NO_BLOCKS = 3,      /* pool exhausted (reject / queue is the caller's policy) */
  PA_ERR_CUDA = 4,           /* a CUDA runtime call failed; see pa_last_error() */
  PA_ERR_DEVICE_BOUNDS = 5,  /* a kernel saw an out-of-range block id / slot / length */
  PA_ERR_DEVICE_TIMEOUT = 6, /* a bounded device-side wait ran out */
  PA_ERR_NOT_FOUND = 7       /* unknown sequence id or block (pool) */
} pa_status;

typedef enum pa_dtype { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* Message describing the last non-zero status returned on this thread. */
PA_API const char* pa_last_error(void);

/* Library ABI version (major * 100 + minor). */
PA_API int pa_version(void);

/* ------------------------------------------------------------------------
 * pa_kv_append -- write the new tokens' K/V rows into their paged slots.
 *
 * OS-lab appendix "Lazy Allocation 与 Copy-on-Write 在 LLM 推理系统中的应用",
 * section 2.1 (each decode step appends the new token's key/value) and the
 * "留书阁 / knowledge-20" page, section "PagedAttention：虚实分离，按需取用"
 * (logical block -> physical block; a token's slot is physical * 16 + offset).
 *
 * For every i < num_tokens with slot_mapping[i] >= 0:
 *   k_cache[slot / 16][h][slot % 16][:] = k[i][h][:]   for all h, likewise v.
 * A negative slot is a padding token and is skipped.  A slot >= num_blocks*16
 * is skipped and sets PA_ERR_DEVICE_BOUNDS.  Bit-exact copy.  Two tokens
 * mapping to the same slot race (the pool never produces that).
 * k, v, k_cache, v_cache must be 16-byte aligned.
 * ---------------------------------------------------------------------- */
PA_API int pa_kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                        int head_dim, int num_blocks, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_workspace_size -- bytes of device workspace that
 * pa_paged_attention_decode needs for these sizes (split partial results,
 * the work list and per-(sequence, KV head) arrival counters).
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_workspace_size(int num_seqs, int num_q_heads,
                                                    int num_kv_heads, int head_dim,
                                                    int max_blocks_per_seq, size_t* bytes);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode -- one decode step of attention over paged K/V.
 *
 * "vLLM: treating the KV cache as virtual memory", sections 破除误解 and
 * "KV 的体积从哪来，页表如何把它切开" (loop over blocks doing Q x K/V
 * multiply-add, then reduce across blocks); "留书阁 / knowledge-20" page,
 * section 注意力计算的改写 (the contiguous reference softmax(QK^T/sqrt(d))V).
 *
 * For each sequence b and query head h, with G = num_q_heads/num_kv_heads,
 * g = h / G, n = context_lens[b] and phys(t) = block_tables[b][t / 16]:
 *   s_t = scale * q[b][h] . k_cache[phys(t)][g][t % 16],  t < n
 *   out[b][h] = sum_t softmax(s)_t * v_cache[phys(t)][g][t % 16]
 * n == 0 gives a zero row.  Accumulation is fp32 (bf16/fp16 inputs use the
 * tensor cores for the two contractions, the probabilities are rounded to the
 * input type before the P.V product); fp32 inputs run on the CUDA cores.
 * Results do not depend on where the blocks sit physically.
 *
 * Preconditions checked on the host: G in 1..8 for F16/BF16 (any G for F32),
 * head_dim in {64, 128}, 16-byte aligned tensors, workspace_bytes at least
 * the size pa_paged_attention_decode_workspace_size() reports.  Checked on
 * the device: 0 <= n <= max_blocks_per_seq * 16 and every table entry read
 * in [0, num_blocks) -- a violation is clamped and sets PA_ERR_DEVICE_BOUNDS.
 *
 * Slots of the last block past the context are never read into the result,
 * whatever they hold (NaN included).
 *
 * The workspace belongs to one call at a time: two calls sharing it must be
 * ordered on the same stream.  It needs no initialisation.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int max_blocks_per_seq, int num_blocks,
                                     float scale, int dtype, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_plan / pa_paged_attention_decode_run -- the same
 * computation as pa_paged_attention_decode, split so that one plan serves
 * every layer of a decode step.
 *
 * The plan (a one-block kernel) turns context_lens into the work list of the
 * attention kernel and stores it in the workspace; it depends only on the
 * context lengths and the shapes, which are the same for every layer of a
 * step ("vLLM: treating the KV cache as virtual memory", section
 * 调度：词一级的进入与退出: one scheduling decision per generated token).
 * Any number of runs may follow one plan, in stream order, with the same
 * context_lens values, num_seqs, head counts, head_dim, max_blocks_per_seq and
 * workspace; each run leaves the workspace ready for the next.  A run whose
 * workspace holds no plan for its shapes does nothing and sets the status
 * word (pa_check_status returns PA_ERR_INVALID_ARG).  After a run that timed
 * out, plan again.  F32 runs do not use the plan.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_plan(const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq, void* workspace,
                                          size_t workspace_bytes, void* stream);
PA_API int pa_paged_attention_decode_run(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int max_blocks_per_seq, int num_blocks,
                                         float scale, int dtype, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_append_run -- pa_kv_append of one new token per
 * sequence followed by pa_paged_attention_decode_run, in one launch.
 *
 * The two steps of a decode step the OS-lab appendix, section 2.1, describes
 * for every layer (append the new token's K/V, then attend over the whole
 * context including it), fused: the pages do not fuse them, the result is the
 * same bit for bit.
 *
 * Row b of k_new / v_new ([num_seqs][num_kv_heads][head_dim], q's dtype) is
 * sequence b's new token.  It is stored at slot_mapping[b] (int64, device)
 * exactly as pa_kv_append stores token b, and sequence b attends over its
 * context_lens[b] tokens, the last of which is the new one: slot_mapping[b]
 * must be block_tables[b][(L - 1) / 16] * 16 + (L - 1) % 16 with
 * L = context_lens[b] > 0, or negative (no new token: the row is not stored
 * and the cache is attended as it is).  A slot >= num_blocks * 16, or one that
 * is not that position, sets PA_ERR_DEVICE_BOUNDS (an out-of-range slot is
 * not stored; for the other, sequence b's output is unspecified).  The block
 * holding the new token must not be read by another sequence of the batch
 * (copy-on-write guarantees this).  For context_lens[b] == 0 the row is
 * stored and the output row is zero.  Needs a plan in the workspace like
 * pa_paged_attention_decode_run.  F32 runs the two steps as two launches.
 * Arguments otherwise as pa_paged_attention_decode_run; k_cache / v_cache
 * are written.  k_new and v_new must be 16-byte aligned.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_append_run(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
    int num_blocks, float scale, int dtype, void* out, void* workspace, size_t workspace_bytes,
    void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_shared_prefix -- pa_paged_attention_decode for a
 * batch whose block tables all start with the same prefix_blocks blocks (a
 * shared system prompt): the prefix's K/V are read once for all queries.
 *
 * "vLLM: treating the KV cache as virtual memory", section 碎片从哪里来 and
 * "第 6 章 缓存管理", section 块表长什么样 (sequences sharing a prefix point
 * their tables at the same physical blocks); the merge of the two parts is
 * the same log-sum-exp reduction across blocks as the split merge ("KV
 * 的体积从哪来，页表如何把它切开": reduce across blocks).  Reading the shared
 * blocks once per batch instead of once per sequence is our extension.
 *
 * Same result and arguments as pa_paged_attention_decode, plus prefix_blocks
 * (0 .. max_blocks_per_seq): every sequence's block_tables[b][0 ..
 * prefix_blocks - 1] must equal row 0's and context_lens[b] >= prefix_blocks
 * * 16 (a violation sets PA_ERR_DEVICE_BOUNDS; that sequence's output is then
 * unspecified).  Three phases on `stream`: the prefix (all queries against
 * the shared blocks, a CTA-shared K/V ring, tensor cores), each sequence's
 * own blocks (the decode kernel), and a log-sum-exp merge.  (With the
 * environment variable PA_CASCADE=grouped, read once per process, it runs
 * as the one-group case of pa_paged_attention_decode_grouped_prefix
 * instead.)  Workspace:
 * pa_paged_attention_decode_shared_prefix_workspace_size bytes.
 * prefix_blocks == 0 or F32 runs a plain decode.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_shared_prefix_workspace_size(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
    size_t* bytes);
PA_API int pa_paged_attention_decode_shared_prefix(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int prefix_blocks, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_shared_prefix_plan / _run -- the plans and the
 * compute launches of pa_paged_attention_decode_shared_prefix as separate
 * calls, so that one plan serves every layer of a decode step.  (No
 * counterpart on the pages: the split exists for callers, not for the
 * method.)
 *
 * _plan reads only context_lens (device) and the sizes, and launches the two
 * work-list plans (the prefix phase's and the suffix decode's) into the
 * workspace; scale and dtype pick the kernels the lists are cut for.  _run
 * takes pa_paged_attention_decode_shared_prefix's arguments and launches the
 * prefix phase, the suffix decode and the combine.  It needs a plan made with
 * the same sizes, prefix_blocks, dtype and sign of scale and the same
 * context_lens contents, in stream order on the same workspace; in a run
 * whose workspace holds no plan for its sizes the attention kernels do
 * nothing and set the status word (pa_check_status returns
 * PA_ERR_INVALID_ARG), and out is unspecified; changed lengths under the
 * same sizes are not detected and give unspecified output.  Runs may
 * follow one plan any number of times; each leaves the workspace ready for
 * the next.  With prefix_blocks == 0 the pair is the plain decode's plan and
 * run; for PA_F32 the plan does nothing.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_shared_prefix_plan(
    const int32_t* context_lens, int prefix_blocks, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, float scale, int dtype,
    void* workspace, size_t workspace_bytes, void* stream);
PA_API int pa_paged_attention_decode_shared_prefix_run(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int prefix_blocks, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_grouped_prefix -- pa_paged_attention_decode for
 * a batch made of groups of sequences, each group sharing its own prefix
 * (the branches of one prompt forked for parallel sampling, requests that
 * share one of several system prompts): every group's prefix is read once
 * for all of the group's queries.
 *
 * "第 6 章 缓存管理", section 块表长什么样, and the OS-lab appendix, section
 * 4.3 (forked sequences point their tables at the same physical blocks until
 * a write copies one); the merge is the log-sum-exp reduction across blocks
 * of "KV 的体积从哪来，页表如何把它切开".  Reading a group's shared blocks
 * once per group is our extension, as in the single-prefix form above.
 *
 * Same result and arguments as pa_paged_attention_decode, plus:
 *   group_start          DEVICE int32 [num_groups + 1]: group g is sequences
 *                        group_start[g] .. group_start[g + 1] - 1 (members
 *                        of a group are contiguous in the batch);
 *                        group_start[0] = 0, group_start[num_groups] =
 *                        num_seqs, non-decreasing.
 *   group_prefix_blocks  DEVICE int32 [num_groups]: how many leading table
 *                        entries every member of group g shares with the
 *                        group's first member (0 .. max_blocks_per_seq; 0:
 *                        nothing shared).  A member's context must cover
 *                        them (context_lens[b] >= 16 * group_prefix_blocks).
 *   num_groups           1 .. num_seqs.
 * A member whose table does not start with its group's prefix, or whose
 * group data or length is out of range, sets the status word
 * (PA_ERR_DEVICE_BOUNDS from pa_check_status); its output is then
 * unspecified.  16-bit dtypes only (PA_F32 returns PA_ERR_UNSUPPORTED: the
 * fp32 decode is exact without it).  The workspace holds
 * pa_paged_attention_decode_grouped_prefix_workspace_size bytes (256-byte
 * aligned).
 *
 * _plan (block_tables, context_lens and the group arrays; once per decode
 * step) checks the groups and writes the work list into the workspace; _run
 * (per layer, same sizes and arrays, same workspace, stream order) launches
 * the attention, which also merges each sequence's splits.  The work list
 * has units of two kinds: a split of a group's shared blocks for up to 16
 * query rows of its members (16 / (num_q_heads / num_kv_heads) members,
 * every shared block read once for them), and a split of one sequence's
 * blocks past the shared ones; a chunk of at most 4 members with at most 16
 * blocks of its own in all takes those into its last shared split instead.
 * (With the environment variable PA_CASCADE=phases, read once per process,
 * the entry points use the three launches of the single-prefix form
 * instead: prefix phase, suffix decode, combine.)  In a run whose workspace
 * holds no plan for its sizes the attention kernel does nothing and sets
 * the status word (PA_ERR_INVALID_ARG), and out is unspecified; tables or
 * lengths changed after the plan are not detected and give unspecified
 * output.  The one-shot entry is _plan then _run.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_grouped_prefix_workspace_size(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
    size_t* bytes);
PA_API int pa_paged_attention_decode_grouped_prefix(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* group_start, const int32_t* group_prefix_blocks,
    int num_groups, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* out, void* workspace,
    size_t workspace_bytes, void* stream);
PA_API int pa_paged_attention_decode_grouped_prefix_plan(
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* group_start,
    const int32_t* group_prefix_blocks, int num_groups, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, float scale, int dtype,
    void* workspace, size_t workspace_bytes, void* stream);
PA_API int pa_paged_attention_decode_grouped_prefix_run(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* group_start, const int32_t* group_prefix_blocks, int num_groups, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
    float scale, int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_shared_prefix_append_run,
 * pa_paged_attention_decode_grouped_prefix_append_run -- the _run of the
 * single-prefix and grouped forms above with the step's new K/V rows stored
 * and attended in the same launches, as pa_paged_attention_decode_append_run
 * does for the plain decode (OS-lab appendix, section 2.1: each decode step
 * appends the new token's key/value).
 *
 * k_new, v_new: [num_seqs][num_kv_heads][head_dim] (16-byte aligned);
 * slot_mapping: DEVICE int64 [num_seqs], sequence b's new slot
 * (physical * 16 + offset), < 0 for none.  Same result as pa_kv_append of
 * the rows followed by the _run.  The new token of sequence b must be the last
 * of its context and lie past the shared prefix, in a block of its own (the
 * copy-on-write pool never appends into a shared block): the prefix phase
 * does not see it.  A slot that is not the position of the sequence's last
 * token, or a sequence with nothing past the prefix that has a slot, sets
 * PA_ERR_DEVICE_BOUNDS.  The plan is the same _plan as above.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_shared_prefix_append_run(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    int prefix_blocks, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* out, void* workspace,
    size_t workspace_bytes, void* stream);
PA_API int pa_paged_attention_decode_grouped_prefix_append_run(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* group_start,
    const int32_t* group_prefix_blocks, int num_groups, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_prefill -- chunked-prefill attention over the paged cache.
 *
 * OS-lab appendix, section 2.1 (prefill writes the K/V of every prompt token
 * into the cache) and "vLLM: treating the KV cache as virtual memory",
 * section "KV 的体积从哪来，页表如何把它切开" (chunked prefill: a long prompt's
 * computation is cut into pieces run between decode steps).
 *
 * Sequence b holds context_lens[b] tokens; its newest T_b tokens are a chunk
 * whose K/V are already in the cache (pa_kv_append) and whose queries are
 * rows query_start[b] .. query_start[b + 1] - 1 of q ([total_q][num_q_heads]
 * [head_dim]); query_start (int32, device, num_seqs + 1 entries) is
 * non-decreasing, query_start[0] >= 0, query_start[num_seqs] <= total_q.
 * Query row i of sequence b is token p = context_lens[b] - T_b + i and, for
 * query head h, attends over tokens 0 .. p with KV head h / (num_q_heads /
 * num_kv_heads):
 *   out[row][h] = softmax_t(scale * q[row][h] . K_t) V_t,  t <= p.
 * T_b = 1 everywhere is decode; T_b = 0 skips the sequence.  out has q's
 * shape and dtype; rows of no sequence are not written.  A sequence with
 * T_b > context_lens[b], context_lens[b] > max_blocks_per_seq * 16 or rows
 * outside [0, total_q) is skipped and sets PA_ERR_DEVICE_BOUNDS, as does a
 * table entry outside [0, num_blocks) (read as block 0).
 *
 * Workspace: pa_paged_attention_prefill_workspace_size bytes, 256-byte
 * aligned, owned by one call at a time, no initialisation needed.  Two
 * launches (a one-CTA plan, then the attention kernel) on `stream`.  Same
 * dtypes, head_dim and grouping limits as pa_paged_attention_decode.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_prefill_workspace_size(int num_seqs, int total_q, int num_q_heads,
                                                     int num_kv_heads, int head_dim,
                                                     size_t* bytes);
PA_API int pa_paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      const int32_t* query_start, int num_seqs, int total_q,
                                      int num_q_heads, int num_kv_heads, int head_dim,
                                      int max_blocks_per_seq, int num_blocks, float scale,
                                      int dtype, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_prefill_plan / pa_paged_attention_prefill_run -- the two
 * launches of pa_paged_attention_prefill as separate calls, so that one plan
 * serves every layer of a model step (the chunks, and so the work list, are
 * the same in every layer).  (No counterpart on the pages: the split exists
 * for callers, not for the method.)
 *
 * _plan reads only context_lens and query_start (device) and the sizes, and
 * writes the work list into the workspace; scale and dtype pick the kernel
 * the work list is cut for.  _run takes pa_paged_attention_prefill's
 * arguments and launches only the attention kernel; it needs a plan made
 * with the same sizes, dtype and sign of scale and with the same
 * context_lens / query_start contents, in stream order on the same
 * workspace.  A run whose workspace holds no plan for its sizes does nothing
 * and sets the status word (pa_check_status returns PA_ERR_INVALID_ARG);
 * changed lengths under the same sizes are not detected and give unspecified
 * output.  Runs may follow one plan any number of times, on any caches,
 * queries and outputs; each leaves the workspace ready for the next.  After
 * a run that timed out, plan again.  For PA_F32 the plan does nothing and
 * the run is the whole call.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_prefill_plan(const int32_t* context_lens,
                                           const int32_t* query_start, int num_seqs,
                                           int total_q, int num_q_heads, int num_kv_heads,
                                           int head_dim, int max_blocks_per_seq, float scale,
                                           int dtype, void* workspace, size_t workspace_bytes,
                                           void* stream);
PA_API int pa_paged_attention_prefill_run(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, const int32_t* context_lens,
                                          const int32_t* query_start, int num_seqs, int total_q,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq, int num_blocks, float scale,
                                          int dtype, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_paged_attention_decode_noalloc -- pa_paged_attention_decode without a
 * caller-provided workspace.  (No counterpart on the pages: this entry point
 * exists for callers, not for the method.)
 *
 * For callers that cannot allocate device memory: code running inside a host
 * framework that owns the whole device-memory budget (a serving engine's
 * pre-reserved pool, a process held to a memory cap) may not call cudaMalloc
 * to make the workspace the other entry point needs.  This one uses a 128 MiB
 * scratch array compiled into the library instead; every GPU that loads the
 * library holds that array until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Same arguments and results as pa_paged_attention_decode, minus the
 * workspace.  Shapes whose workspace (see
 * pa_paged_attention_decode_workspace_size) exceeds 128 MiB are rejected with
 * PA_ERR_INVALID_ARG before anything is launched.  The first call on a device
 * looks up that device's scratch address (cudaGetSymbolAddress, with the
 * device current), so make the first call on each device before any stream
 * capture.  Every call re-plans its work into the scratch, so nothing needs
 * clearing between calls; but all calls on a device share the one array, so
 * two calls whose kernels overlap on the GPU (different streams, no ordering)
 * race and corrupt each other's results.
 * ---------------------------------------------------------------------- */
PA_API int pa_paged_attention_decode_noalloc(const void* q, const void* k_cache,
                                             const void* v_cache, const int32_t* block_tables,
                                             const int32_t* context_lens, int num_seqs,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int max_blocks_per_seq, int num_blocks, float scale,
                                             int dtype, void* out, void* stream);

/* ------------------------------------------------------------------------
 * pa_block_copy -- copy-on-write block copies, all layers in one launch.
 *
 * OS-lab appendix, sections 4.3-4.4 (when the target block's refcount is
 * above one, copy it for the writer first); "第 6 章 缓存管理", section
 * 块表长什么样 (modify a copy, never the shared block).
 *
 * k_caches / v_caches: HOST arrays of num_layers device pointers, each a
 * cache as laid out above.  src_dst_pairs: DEVICE int64 [num_pairs][2].
 * For every pair and layer: k_caches[l][dst] = k_caches[l][src] (the whole
 * num_kv_heads * 16 * head_dim block), likewise v.  Pairs run concurrently:
 * no dst may repeat or appear as another pair's src (the pool's pairs for one
 * step satisfy this).  Ids outside [0, num_blocks) skip that pair and set
 * PA_ERR_DEVICE_BOUNDS.  num_layers <= 256.
 * ---------------------------------------------------------------------- */
PA_API int pa_block_copy(void* const* k_caches, void* const* v_caches, int num_layers,
                         const int64_t* src_dst_pairs, int num_pairs, int num_kv_heads,
                         int head_dim, int num_blocks, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * pa_block_swap -- copy whole blocks between the device caches and caches in
 * page-locked host memory, every layer, in one launch.
 *
 * "vLLM: treating the KV cache as virtual memory", section
 * 调度：词一级的进入与退出 (a preempted sequence's KV is offloaded to host
 * memory and loaded back later, block by block) and "第 6 章 缓存管理",
 * section 缓存放不下的时候 (spill cold cache to CPU memory; a CPU with a fast
 * link to the GPU reaches hundreds of GB/s).
 *
 * direction PA_SWAP_OUT: pairs[i] = (device block, host block) and
 *   host_k[l][host block] = dev_k[l][device block] (likewise v) for every l;
 * direction PA_SWAP_IN: pairs[i] = (host block, device block), the reverse.
 * These are the pairs pa_pool_swap_out / pa_pool_swap_in produce (copied to
 * the device).  Host caches are [num_host_blocks][num_kv_heads][16][head_dim]
 * per layer in page-locked host memory (cudaHostAlloc / cudaHostRegister;
 * anything else is PA_ERR_INVALID_ARG); dev/host cache pointer arrays are
 * host arrays of num_layers (<= 256) pointers; pairs is device memory.
 * Bit-exact.  A block id out of range skips the pair and sets
 * PA_ERR_DEVICE_BOUNDS.  Destinations must be distinct.
 * ---------------------------------------------------------------------- */
#define PA_SWAP_OUT 0
#define PA_SWAP_IN 1
PA_API int pa_block_swap(void* const* dev_k_caches, void* const* dev_v_caches,
                         void* const* host_k_caches, void* const* host_v_caches, int num_layers,
                         const int64_t* pairs, int num_pairs, int direction, int num_kv_heads,
                         int head_dim, int num_dev_blocks, int num_host_blocks, int dtype,
                         void* stream);

/* ------------------------------------------------------------------------
 * pa_check_status -- synchronise `stream`, then read and clear the device
 * status word of the current device.  Returns PA_OK, PA_ERR_DEVICE_BOUNDS,
 * PA_ERR_DEVICE_TIMEOUT, PA_ERR_INVALID_ARG (a decode run found no plan in
 * its workspace), or PA_ERR_CUDA if the synchronisation failed.
 * ---------------------------------------------------------------------- */
PA_API int pa_check_status(void* stream);

/* ========================================================================
 * Host block pool.  Produces block tables, slots and copy-on-write pairs;
 * touches no device memory.  Not thread-safe: one pool per thread or
 * external locking.
 *
 * Semantics ("vLLM: treating the KV cache as virtual memory", section
 * 碎片从哪里来; "第 6 章 缓存管理", section 块表长什么样; OS-lab appendix
 * sections 3.3 and 4.3-4.4; "留书阁 / knowledge-20" page, section
 * 写时复制与前缀缓存):
 *  - free list is a stack; it starts as initial_order (initial_order[0] is
 *    handed out first; NULL = 0, 1, 2, ...);
 *  - a block is taken only when a sequence's next token starts a new logical
 *    block (lazy allocation);
 *  - fork and share_prefix copy table entries and raise refcounts;
 *  - appending into a block whose refcount is above one moves the writer to
 *    a fresh block and reports the (src, dst) pair to copy; the last holder
 *    writes in place;
 *  - a block returns to the free list when its refcount reaches zero, unless
 *    pinned (prefix cache);
 *  - freeing a sequence releases its blocks from the last logical block to
 *    the first; sequence ids count up from 0 and are never reused.
 * ====================================================================== */
typedef struct pa_pool pa_pool;

typedef struct pa_pool_stats_t {
  int64_t num_blocks;
  int64_t free_blocks;
  int64_t used_blocks;         /* refcount > 0 */
  int64_t pinned_blocks;
  int64_t shared_blocks;       /* refcount > 1 */
  int64_t cow_copies;          /* cumulative copy-on-write pairs produced */
  int64_t live_seqs;
  int64_t tokens;              /* sum of live context lengths */
  int64_t internal_frag_slots; /* sum over live seqs of table slots minus tokens */
  int64_t host_blocks;         /* size of the host tier (pa_pool_set_host_blocks) */
  int64_t host_free_blocks;
  int64_t swapped_seqs;        /* live sequences whose blocks are on the host tier */
  int64_t cached_blocks;       /* blocks keyed in the prefix cache */
  int64_t evictable_blocks;    /* keyed blocks nobody holds (LRU list) */
  int64_t prefix_hit_tokens;   /* cumulative prompt tokens served from the cache */
  int64_t evictions;           /* cumulative cached blocks evicted for reuse */
} pa_pool_stats_t;

/* block_size >= 1 (device kernels accept only 16; other sizes serve host
 * bookkeeping).  initial_order: NULL or a permutation of 0..num_blocks-1. */
PA_API int pa_pool_create(int num_blocks, int block_size, const int32_t* initial_order,
                          pa_pool** pool);
PA_API int pa_pool_destroy(pa_pool* pool);
PA_API int pa_pool_new_seq(pa_pool* pool, int* seq_id);
/* Reserve the slot of `seq`'s next token.  *cow_src / *cow_dst receive the
 * block pair to copy before writing, or -1 / -1.  PA_ERR_NO_BLOCKS leaves the
 * pool unchanged. */
PA_API int pa_pool_append_slot(pa_pool* pool, int seq, int64_t* slot, int64_t* cow_src,
                               int64_t* cow_dst);
/* Batched form: one slot per entry of seqs[0..n), written to slots[] and the
 * copy pairs (if any) appended to pairs[] (int64 [*num_pairs][2], capacity
 * pair_cap; pairs may be NULL only when pair_cap == 0).  Stops at the first
 * error; *done tells how many succeeded. */
PA_API int pa_pool_append_slots(pa_pool* pool, const int32_t* seqs, int n, int64_t* slots,
                                int64_t* pairs, int pair_cap, int* num_pairs, int* done);
PA_API int pa_pool_fork(pa_pool* pool, int parent, int* child);
PA_API int pa_pool_share_prefix(pa_pool* pool, int src_seq, int dst_seq, int num_tokens);
PA_API int pa_pool_pin(pa_pool* pool, int seq, int num_tokens);
PA_API int pa_pool_unpin(pa_pool* pool, int block);
PA_API int pa_pool_free_seq(pa_pool* pool, int seq);
/* Copies up to `cap` table entries to out[] (may be NULL when cap == 0);
 * *n receives the full table length and *ctx_len the context length. */
PA_API int pa_pool_block_table(pa_pool* pool, int seq, int32_t* out, int cap, int* n,
                               int* ctx_len);
PA_API int pa_pool_refcount(pa_pool* pool, int block, int* rc);
PA_API int pa_pool_stats(pa_pool* pool, pa_pool_stats_t* stats);

/* Swapping ("vLLM: treating the KV cache as virtual memory", section
 * 调度：词一级的进入与退出: a preempted sequence's KV goes to host memory and
 * comes back later, block by block; "第 6 章 缓存管理", section
 * 缓存放不下的时候: spill cold cache to CPU memory).
 *
 * pa_pool_set_host_blocks gives the pool a host tier of num_host_blocks
 * blocks (a LIFO free list started from initial_order, NULL = identity); it
 * fails while a sequence is swapped out.
 *
 * pa_pool_swap_out moves sequence seq to the host tier: for each logical
 * block i in order it takes a host block and writes the copy pair
 * (device block, host block) to pairs[2i], pairs[2i+1] (host int64 buffer of
 * cap pairs), then releases the device blocks last to first.  *n = number of
 * pairs.  Copy them (pa_block_swap) before the device blocks are written
 * again.  Fails (nothing changed) when a block is shared (refcount > 1) or
 * pinned (PA_ERR_INVALID_ARG), the host tier is short (PA_ERR_NO_BLOCKS) or
 * cap is too small.  pa_pool_swap_in is the mirror image: pairs are
 * (host block, device block), the device blocks come from the free list.
 * A swapped sequence cannot append, fork, share or pin (PA_ERR_INVALID_ARG);
 * its block table reports its host blocks; freeing it returns them. */
PA_API int pa_pool_set_host_blocks(pa_pool* pool, int num_host_blocks,
                                   const int32_t* initial_order);
PA_API int pa_pool_swap_out(pa_pool* pool, int seq, int64_t* pairs, int cap, int* n);
PA_API int pa_pool_swap_in(pa_pool* pool, int seq, int64_t* pairs, int cap, int* n);
PA_API int pa_pool_is_swapped(pa_pool* pool, int seq, int* swapped);

/* Prefix cache ("vLLM: treating the KV cache as virtual memory", section
 * 碎片从哪里来: hot prefixes stay outside the free list so the next request
 * with the same system prompt hits them; "第 6 章 缓存管理", section
 * 缓存放不下的时候: evict in least-recently-used order, recompute next time).
 *
 * pa_pool_enable_prefix_cache must come before the first sequence.  A full
 * block is keyed by 64-bit FNV-1a over its parent block's key (8 bytes LE, 0
 * for a first block) and its block_size token ids (int32 LE); lookups also
 * compare the parent block and the ids, so equal hashes never alias.
 * pa_pool_new_seq_with_prompt creates a sequence for a prompt of n token ids
 * and gives it the longest run of leading full cached blocks (refcount + 1),
 * leaving at least one token to compute: *hit_tokens (a multiple of
 * block_size) tokens are already in the cache, the caller appends the rest.
 * pa_pool_append_token is pa_pool_append_slot for a sequence whose token ids
 * are tracked (made by new_seq_with_prompt, or forked / shared from one): a
 * block it fills is keyed unless that key is already cached.  (A plain
 * pa_pool_append_slot stops the tracking for that sequence.)  A keyed block
 * whose refcount reaches zero joins the LRU list instead of the free list;
 * allocations take the free list first and evict the least recently used
 * cached block only when it is empty.  Stats report cached and evictable
 * blocks, hit tokens and evictions. */
PA_API int pa_pool_enable_prefix_cache(pa_pool* pool, int on);
PA_API int pa_pool_new_seq_with_prompt(pa_pool* pool, const int32_t* tokens, int n, int* seq_id,
                                       int* hit_tokens);
PA_API int pa_pool_append_token(pa_pool* pool, int seq, int32_t token, int64_t* slot,
                                int64_t* cow_src, int64_t* cow_dst);
/* Batched form of pa_pool_append_token, for a serving loop that adds one
 * token to every running sequence each step ("留书阁 / knowledge-20" page,
 * section on continuous batching): token tokens[i] appended to sequence
 * seqs[i] for i = 0, 1, ... in order (a sequence may repeat: a prompt's
 * tokens), slots to slots[], copy pairs appended to pairs[] (int64
 * [*num_pairs][2], capacity pair_cap; NULL only when pair_cap == 0).  Stops
 * at the first failing append and
 * returns its status (PA_ERR_NO_BLOCKS when the pool ran out) with *done =
 * the appends made; a full pair buffer returns PA_ERR_INVALID_ARG before the
 * append that would need it. */
PA_API int pa_pool_append_tokens(pa_pool* pool, const int32_t* seqs, const int32_t* tokens,
                                 int n, int64_t* slots, int64_t* pairs, int pair_cap,
                                 int* num_pairs, int* done);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
