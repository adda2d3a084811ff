// TMA tensor maps over a paged K or V cache, shared by the attention kernels.
#pragma once

#include <cuda.h>

namespace pa {

// Encodes (or takes from a per-thread cache) the 2-D tensor map of one cache
// `[num_blocks][num_kv_heads][16][head_dim]` of 16-bit elements: rows =
// num_blocks * num_kv_heads * 16 token rows of head_dim elements, one copy
// box = 16 rows x 64 elements (128 bytes wide, 128-byte swizzle), so a
// (block, head) tile is head_dim / 64 boxes.  In shared memory box h of a
// tile sits at h * 2048, row r at r * 128, its 16-byte chunks XOR-swizzled by
// r % 8.  A decode or prefill step reuses the same layer caches every step and
// encoding is a host-side driver call, hence the cache.  Returns a pa_status.
int cache_tensor_map(CUtensorMap* out, const void* cache, bool bf16, int num_blocks,
                     int num_kv_heads, int head_dim);

// Encodes the 3-D tensor map of a query tensor `[total_q][num_q_heads][head_dim]`
// (16-bit) whose copy box is 64 elements x `group` heads x (rows / group)
// tokens with 128-byte swizzle: one box fills `rows` consecutive 128-byte
// rows of a query tile, row = token * group + head within the group.
// Returns a pa_status.
int query_tensor_map(CUtensorMap* out, const void* q, bool bf16, int total_q, int num_q_heads,
                     int head_dim, int group, int rows);

// Encodes the 3-D tensor map of an output tensor `[total_q][num_q_heads]
// [head_dim]` (16-bit) for stores whose box is 64 elements x `group` heads x
// (rows / group) tokens with 128-byte swizzle: in shared memory the box's
// `rows` rows of 128 bytes sit one after another (row = token * group + head
// within the group), the 16-byte chunk c of row r at chunk c ^ (r % 8).
// Returns a pa_status.
int output_tensor_map(CUtensorMap* out, void* o, bool bf16, int total_q, int num_q_heads,
                      int head_dim, int group, int rows);

}  // namespace pa
