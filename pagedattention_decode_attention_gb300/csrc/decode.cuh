// Shared definitions between the decode kernels and their host launcher.
#pragma once

#include <cstddef>
#include <cstdint>

namespace pa {
namespace decode {

constexpr int kBlockSize = 16;      // tokens per physical block (device kernels)
constexpr int kSplitBlocks = 32;    // most logical blocks per work item (512 tokens)
constexpr int kMinSplitBlocks = 16; // fewest blocks a split may be planned with
constexpr int kPieceBlocks = 8;     // default: most blocks of a piece at the end of the work list
constexpr int kTailWaves = 1;       // pieces at the end: about this many per math warp
constexpr int kConsumerWarps = 8;   // default number of math warps per CTA
constexpr int kWarpStages = 4;      // upper bound of each math warp's (K, V) tile ring
constexpr int kMaxGroup = 8;        // query heads per KV head on the tensor-core path

// Workspace header words.
constexpr int kHdrNext = 0;       // next work item (self-resetting)
constexpr int kHdrTotal = 1;      // number of work items (written by the plan)
constexpr int kHdrDone = 2;       // warps that have taken their last item (self-resetting)
constexpr int kHdrSignature = 3;  // shape signature written by the plan
// grouped decode: its merges go through a queue in the attention launch
constexpr int kHdrQHead = 4;      // next queue entry to take (self-resetting)
constexpr int kHdrQTail = 5;      // next queue entry to fill (self-resetting)
constexpr int kHdrQDone = 6;      // warps done with the queue (self-resetting)
constexpr int kHdrMerges = 7;     // merges the run will queue (written by the plan)
// grouped decode: kTeamWarps when the plan placed its units in teams (the
// splits of one (chunk, KV head) on kTeamWarps warps of one CTA, merged in
// shared memory), else 0 (merges through the queue)
constexpr int kHdrTeam = 8;
constexpr int kTeamWarps = 4;

// Views into the caller's workspace (all offsets 256-byte aligned).
struct Workspace {
  int* header;       // see kHdr*
  // int4 per unit: (b, first block, split index << 16 | members << 8 | blocks,
  // ctx); members is 0 for a unit of one sequence, else the number of
  // consecutive sequences from b that share the unit's blocks (grouped plan)
  int* units;
  int* arrivals;     // [num_seqs * num_kv_heads] finished splits per (b, kv head)
  int* nsplits;      // [num_seqs] splits the plan made of each sequence
  float* part_lse;   // [num_seqs][max_splits][num_q_heads]  (log2 domain)
  float* part_o;     // [num_seqs][max_splits][num_q_heads][head_dim]
  // grouped decode only (else null): [num_seqs * num_kv_heads] queue of
  // merges, entry i = 1 + (b * num_kv_heads + g) once (b, g) is ready, 0 before
  int* mqueue;
};

struct Layout {
  size_t header, units, arrivals, nsplits, part_lse, part_o, total;
  int max_splits;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline Layout workspace_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int max_blocks_per_seq) {
  Layout l;
  // sized for the smallest split the plan may choose
  l.max_splits = int((int64_t(max_blocks_per_seq) + kMinSplitBlocks - 1) / kMinSplitBlocks);
  if (l.max_splits < 1) l.max_splits = 1;
  const size_t units = size_t(num_seqs) * l.max_splits;
  l.header = 0;
  l.units = align256(l.header + 256);
  l.arrivals = align256(l.units + units * 16);
  l.nsplits = align256(l.arrivals + size_t(num_seqs) * num_kv_heads * 4);
  l.part_lse = align256(l.nsplits + size_t(num_seqs) * 4);
  l.part_o = align256(l.part_lse + units * num_q_heads * 4);
  l.total = align256(l.part_o + units * num_q_heads * size_t(head_dim) * 4);
  return l;
}

// True when the workspace of these shapes (with the shared-prefix and
// grouped additions on top) would come near the range of size_t.  The
// layouts multiply the sizes in size_t, so such shapes are rejected before
// any layout is computed; a real device holds far less than the 2^50 bytes
// allowed here.
inline bool layout_too_large(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int max_blocks_per_seq) {
  const double splits = (double(max_blocks_per_seq) + kMinSplitBlocks - 1) / kMinSplitBlocks;
  const double units = double(num_seqs) * (splits < 1.0 ? 1.0 : splits);
  const double rows = double(num_seqs) * num_q_heads;
  const double bytes = units * (16.0 + num_q_heads * (head_dim + 1.0) * 4.0) +
                       double(num_seqs) * (2.0 * num_kv_heads + 2.0) * 4.0 +
                       double(num_seqs) * max_blocks_per_seq * 4.0 +
                       16.0 * rows * (head_dim + 1.0) * 4.0 + 65536.0;
  return bytes > double(uint64_t(1) << 50);
}

// Identifies the shapes a plan was made for, so a run can refuse a workspace
// planned for something else.
inline int plan_signature(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int max_blocks_per_seq, int split_blocks, int table_offset = 0,
                          int grouped = 0) {
  uint32_t h = 2166136261u;
  const int v[8] = {num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                    split_blocks, table_offset, grouped};
  for (int x : v) {
    h ^= uint32_t(x);
    h *= 16777619u;
  }
  return int(h | 1u);
}

struct Params {
  const void* q;
  const void* k_cache;  // raw cache pointers (the fp32 path reads them directly;
  const void* v_cache;  // the tensor-core path goes through tensor maps)
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  // Grouped mode (non-null): per sequence, the leading blocks it shares with
  // its group (written by the grouped plan).  verify_prefix: the run checks
  // that every table starts with sequence 0's seq_prefix[b] entries (the
  // plan of a single shared prefix does not see the tables).
  const int32_t* seq_prefix;
  int verify_prefix;
  // Fused append (all three null: none).  Row b of k_new / v_new
  // ([num_seqs][num_kv_heads][head_dim]) is sequence b's new token, stored at
  // slot_mapping[b] and attended as its token context_lens[b] - 1.
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  // Suffix mode (cas_o non-null): each sequence attends only its tokens from
  // ctx_offset on (table entries from table_offset on), and the results go
  // to cas_o / cas_lse (fp32 o and base-2 log-sum-exp per (sequence, head))
  // for a later merge with the shared prefix's, instead of out.
  int table_offset, ctx_offset;
  float* cas_o;      // [num_seqs * num_q_heads][head_dim]
  float* cas_lse;    // [num_seqs * num_q_heads]
  int num_seqs, num_q_heads, num_kv_heads, group, head_dim;
  int max_blocks, num_blocks, max_splits;
  int stages;        // depth of the shared-memory tile ring (tensor-core path)
  int split_blocks;  // blocks per split, kMinSplitBlocks .. kSplitBlocks
  int tail_blocks;   // plan: work (in blocks) at the end of the list cut into pieces
  int piece_blocks;  // plan: most blocks of such a piece
  int signature;     // plan_signature() of these shapes
  float scale;       // softmax scale (fp32 path)
  float scale_log2;  // scale * log2(e) (tensor-core path works in base 2)
  Workspace ws;
  unsigned* status;
  unsigned long long timeout_ns;
};

}  // namespace decode
}  // namespace pa
