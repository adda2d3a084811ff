// Internal interface of the prefill engine used by other parts of the library.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace pa {
namespace prefill {

// Most (o, lse) parts per row the shared-prefix phase leaves for the caller
// to merge (it splits the prefix into at most this many pieces).
constexpr int kSharedMaxSplits = 8;

// Device address of the word in a shared-prefix phase workspace holding how
// many parts per row the last planned phase leaves (1 .. kSharedMaxSplits).
const int* shared_prefix_split_count(const void* workspace);

// Device address of the word holding the split size in blocks behind those
// parts (0: one part per row); a group of nb prefix blocks then leaves
// shared_prefix_parts(nb, word) parts per row.
const int* shared_prefix_split_blocks(const void* workspace);
__host__ __device__ inline int shared_prefix_parts(int nb, int split_blocks) {
  if (nb <= 0) return 0;
  if (split_blocks <= 0) return 1;
  const int n = (nb + split_blocks - 1) / split_blocks;
  return n < kSharedMaxSplits ? n : kSharedMaxSplits;
}

// Workspace bytes of the shared-prefix phase for a batch of num_seqs decode
// queries (single prefix, or up to num_seqs groups).
size_t shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim);

// Shared-prefix phase of a cascade decode: each of the num_seqs decode
// queries q[b][h] attends all prefix_tokens tokens of the prefix whose blocks
// are block_tables[0][0 ..] (no causal mask); writes fp32 o and the base-2
// log-sum-exp per (sequence, head) to cas_o / cas_lse, as n parts (n the
// word at shared_prefix_split_count, parts k at cas_o + k * rows * head_dim
// and cas_lse + k * rows, rows = num_seqs * num_q_heads) whose log-sum-exp
// merge is the result; cas_o / cas_lse hold kSharedMaxSplits parts.  Two launches (plan +
// kernel) on `stream`.  Returns a pa_status.  16-bit dtypes only.
int shared_prefix_phase(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int prefix_tokens, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                        int num_blocks, float scale, int dtype, float* cas_o, float* cas_lse,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

// The two launches of shared_prefix_phase as separate calls: the plan depends
// only on the sizes and prefix_tokens, so one serves every layer; the run
// needs a plan for the same sizes and prefix_tokens in the workspace.
int shared_prefix_plan(int prefix_tokens, int num_seqs, int num_q_heads, int num_kv_heads,
                       int head_dim, int max_blocks_per_seq, float scale, int dtype,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);
int shared_prefix_run(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int prefix_tokens, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                      int num_blocks, float scale, int dtype, float* cas_o, float* cas_lse,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

// Grouped shared-prefix phase: group g is the decode queries (sequences)
// group_start[g] .. group_start[g + 1] - 1, whose tables all start with the
// same group_blocks[g] blocks (those of sequence group_start[g]); each query
// attends its group's prefix (no causal mask).  group_start / group_blocks
// are device arrays of num_groups + 1 / num_groups entries.  Results as in
// shared_prefix_phase, with each row's part count shared_prefix_parts(nb of
// its group, the word at shared_prefix_split_blocks).  Plan once per step,
// run per layer, as above.
int grouped_prefix_plan(const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_blocks_per_seq, float scale, int dtype, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);
int grouped_prefix_run(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* group_start,
                       const int32_t* group_blocks, int num_groups, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                       float scale, int dtype, float* cas_o, float* cas_lse, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

}  // namespace prefill
}  // namespace pa
