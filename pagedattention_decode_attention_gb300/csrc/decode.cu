// Paged decode attention for sm_103a.
//
// What it computes: for each sequence b and query head h (KV head g = h / G),
//   out[b][h] = softmax_t(scale * q[b][h] . K_t) . V_t,   t < context_lens[b],
// where token t of the sequence lives in physical block block_tables[b][t/16]
// at offset t % 16 ("vLLM: treating the KV cache as virtual memory", section
// 破除误解: the formula is unchanged, the kernel follows the block table with
// one indirection per block; "留书阁 / knowledge-20" page, section
// 注意力计算的改写: per-block multiply-add then a reduction across blocks).
//
// Design (ours; the pages give no kernel design):
//  * plan kernel (1 CTA): splits every sequence into work items of up to
//    kSplitBlocks logical blocks (512 tokens), one item per (sequence, KV
//    head, split); full items first, then partial ones by decreasing size, so
//    the tail of the persistent kernel is made of the smallest items.  The
//    plan depends only on the context lengths, so one plan serves every layer
//    of a decode step.
//  * persistent attention kernel, one CTA of W math warps per SM.  Each warp
//    works alone: it claims whole work items from a global counter (its first
//    item is dealt statically: W consecutive items per CTA, or round robin over
//    the SMs when the list is shorter than the warps, so that it still spreads
//    over every SM), and streams every block of them through its own small ring,
//    issuing the 2-D tensor copies (128-byte swizzled, L2 evict-first) of a
//    block's K and V tiles a few blocks before it needs them.  The claim of the
//    next item is pipelined over the last blocks of the current one (counter
//    reply, work unit, block-table entries with one entry per lane, then a bulk
//    copy of the G query rows), so a warp commits to an item only shortly before
//    it starts it and the work left in the list goes to whichever warp frees up
//    first.  Many independent issuers keep HBM busy; a single issuing thread per
//    CTA could not (each copy instruction costs it hundreds of cycles), and no
//    CTA-wide barrier is needed.  Per 16-token block: S^T = K . Q^T on the
//    tensor cores (m16n8k16, M = the 16 tokens, N = the G <= 8 query heads of
//    the group, K = head_dim), online softmax in base 2 with per-head running
//    max / sum, P rounded to the input type and transposed in registers
//    (movmatrix), O^T += V^T . P^T (M = head_dim rows of V^T via
//    ldmatrix.trans).  Each K/V tile is read from HBM once for the whole query
//    group.  Slots past the context in the last block are zeroed in registers,
//    so whatever bits they hold cannot reach the output.
//    A sequence with one split is written to `out` straight from the
//    warp's registers; otherwise the warp writes (o, lse) to the workspace,
//    publishes it (fence) and counts it (atomic), and the warp that completes
//    the last split of (b, g) merges all splits with log-sum-exp weights (no
//    spinning).  The work and arrival counters return to zero by the end of
//    every run.
//  * Every wait is an mbarrier wait with a time limit; running out sets the
//    timeout bit of the device status word and the warp returns.
//  * Grouped decode (sequences in groups that share leading blocks): the same
//    kernel with two row tiles per item (up to 16 query rows: G heads of up
//    to 16 / G members of a group), planned by grouped_plan_kernel.  A shared
//    unit reads a split of the group's shared blocks once for its members'
//    rows; an own unit covers one sequence's blocks past them; a small chunk
//    takes its members' own blocks into its last shared unit, each block's
//    scores masked to its member's rows.  A member's last split to finish
//    queues the member's merge; warps that have run out of items take the
//    queued merges, in the same launch.
//
// An fp32 path (CUDA cores, one warp per (sequence, head), online softmax in
// natural base) serves float32 caches; it is exact to fp32 rounding and is not
// tuned for speed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "decode.cuh"
#include "trace.h"
#include "device_common.cuh"
#include "pagedattn.h"
#include "prefill.h"
#include "status.h"
#include "tensor_map.h"

namespace pa {
namespace decode {

using dev::mbar_arrive;
using dev::mbar_wait_bounded;

// Optional timestamps per warp and per item, compiled in only with
// -DPA_PROFILE_TIMES (a separate build used to see where a persistent warp
// spends its time; the default build has none of it).
#ifdef PA_PROFILE_TIMES
// per (CTA, warp): globaltimer at start of work, at end, blocks consumed
__device__ unsigned long long g_times[2048 * 16 * 3];
#define TIME_MARK(i, v)                                                                     \
  do {                                                                                      \
    if ((threadIdx.x & 31) == 0)                                                            \
      g_times[(blockIdx.x * 16 + (threadIdx.x >> 5)) * 3 + (i)] = (v);                      \
  } while (0)
// per (CTA, warp): its last 16 items as (start, end, blocks << 32 | splits,
// ns spent merging << 32 | ns waiting for the query rows)
__device__ unsigned long long g_item_trace[2048 * 16 * 16 * 4];
#define ITEM_TRACE(n, start, blocks, splits, merge_ns, qwait_ns)                            \
  do {                                                                                      \
    if ((threadIdx.x & 31) == 0) {                                                          \
      unsigned long long* r_ =                                                              \
          &g_item_trace[((blockIdx.x * 16 + (threadIdx.x >> 5)) * 16 + ((n) & 15)) * 4];    \
      r_[0] = (start);                                                                      \
      r_[1] = dev::global_timer_ns();                                                       \
      r_[2] = (static_cast<unsigned long long>(blocks) << 32) | unsigned(splits);           \
      r_[3] = (static_cast<unsigned long long>(merge_ns) << 32) | unsigned(qwait_ns);       \
    }                                                                                       \
  } while (0)
#else
#define TIME_MARK(i, v)
#define ITEM_TRACE(n, start, blocks, splits, merge_ns, qwait_ns)
#endif

template <int D, int W, int NT>
struct Smem {
  static constexpr int kTileBytes = kBlockSize * D * 2;  // one (block, head) tile
  static constexpr int kStageBytes = 2 * kTileBytes;     // K tile + V tile
  // one warp's staging buffer: its item's query rows (up to 8 NT), and the
  // new token's K row and V row when the item carries the append (after row
  // 7: an item with an append has at most 8 query rows).  With one row tile
  // the rows are kQRow elements apart (16 bytes of padding), so the lanes
  // that read the same head_dim columns of different rows hit different
  // banks; with two the padding would cost the third ring stage.
  static constexpr int kQRow = NT == 1 ? D + 8 : D;
  static constexpr int kQBytes = NT == 1 ? (8 * kQRow + 2 * D) * 2 : 16 * kQRow * 2;
  // layout: rings [W][stages][stage] | query buffers [W] | barriers [W][stages + 1]
  // | team barriers [W / kTeamWarps]
  static constexpr size_t kFixedBytes = 1024 /* alignment slack */ + size_t(W) * kQBytes +
                                        size_t(W) * (kWarpStages + 1) * 8 +
                                        size_t(W / kTeamWarps + 1) * 8;
  static size_t bytes(int stages) { return kFixedBytes + size_t(W) * stages * kStageBytes; }
  // deepest ring (stages per warp) that fits in `budget` bytes
  static int stages_for(size_t budget) {
    const long avail = long(budget) - long(kFixedBytes);
    long st = avail / (long(W) * kStageBytes);
    if (st > kWarpStages) st = kWarpStages;
    return int(st);
  }
};

// ------------------------------------------------------------------ plan
// Splits of one sequence are balanced: nsplit = ceil(blocks / split) splits
// whose sizes differ by at most one block.
__device__ __forceinline__ void split_shape(int nblk, int split, int& nsplit, int& base,
                                            int& big) {
  nsplit = (nblk + split - 1) / split;
  base = nsplit ? nblk / nsplit : 0;
  big = nsplit ? nblk - base * nsplit : 0;  // the first `big` splits hold base + 1 blocks
}

// Units a split of n blocks becomes: itself, or balanced pieces of at most
// `piece` blocks when n <= cut.
__device__ __forceinline__ int pieces_of(int n, int cut, int piece) {
  return n <= cut ? (n + piece - 1) / piece : 1;
}

// The work list is sorted by size, largest first, so the last items the
// persistent kernel hands out are the smallest (longest-processing-time-first
// order).  Its tail is made finer still: the smallest splits, whose work adds
// up to about kTailWaves pieces per math warp, are cut into pieces of at most
// kPieceBlocks blocks (both tunable), so the warps run out of work at nearly
// the same time.
// A sequence is cut only while its units fit the workspace's max_splits.
constexpr int kPlanThreads = 256;  // small enough to sit beside an attention CTA

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const Params p) {
  __shared__ int hist[kSplitBlocks + 2];
  __shared__ int bucket[kSplitBlocks + 2];
  __shared__ int cut_s;
  dev::grid_launch_dependents();
  // the previous kernel may still read the workspace (or write context_lens)
  dev::grid_dependency_wait();
  const int tid = threadIdx.x;
  if (tid < kSplitBlocks + 2) hist[tid] = 0;
  __syncthreads();
  const int cap = (p.max_blocks - p.table_offset) * kBlockSize;
  int4* units = reinterpret_cast<int4*>(p.ws.units);

  // pass 1: split sizes before any cut
  for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
    int ctx = p.context_lens[b] - p.ctx_offset;
    if (ctx < 0 || ctx > cap) {
      dev::flag_status(p.status, kStatusBounds);
      ctx = ctx < 0 ? 0 : cap;
    }
    int nsplit, base, big;
    split_shape((ctx + kBlockSize - 1) / kBlockSize, p.split_blocks, nsplit, base, big);
    if (big) atomicAdd(&hist[base + 1], big);
    if (nsplit - big) atomicAdd(&hist[base], nsplit - big);
    for (int g = 0; g < p.num_kv_heads; ++g) p.ws.arrivals[size_t(b) * p.num_kv_heads + g] = 0;
  }
  __syncthreads();
  if (tid == 0) {
    // largest size `cut` such that all splits of at most `cut` blocks hold no
    // more than the tail's share of the work
    const long long budget = p.tail_blocks / p.num_kv_heads;
    long long acc = 0;
    int cut = 0;
    while (cut < kSplitBlocks && acc + (long long)hist[cut + 1] * (cut + 1) <= budget) {
      ++cut;
      acc += (long long)hist[cut] * cut;
    }
    cut_s = cut;
  }
  __syncthreads();
  const int cut_all = cut_s;
  if (tid < kSplitBlocks + 2) hist[tid] = 0;
  __syncthreads();

  // pass 2: sizes of the final units (splits and pieces)
  for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
    int ctx = p.context_lens[b] - p.ctx_offset;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    int nsplit, base, big;
    split_shape((ctx + kBlockSize - 1) / kBlockSize, p.split_blocks, nsplit, base, big);
    int cut = cut_all;
    if (big * pieces_of(base + 1, cut, p.piece_blocks) + (nsplit - big) * pieces_of(base, cut, p.piece_blocks) > p.max_splits)
      cut = 0;
    int count = 0;
    for (int k = 0; k < 2; ++k) {  // the two split sizes
      const int n = base + 1 - k, m = k ? nsplit - big : big;
      if (m == 0 || n == 0) continue;
      const int np = pieces_of(n, cut, p.piece_blocks);
      count += m * np;
      const int pb = n / np, pr = n - pb * np;  // pr pieces of pb + 1, the rest of pb
      if (pr) atomicAdd(&hist[pb + 1], m * pr);
      if (np - pr) atomicAdd(&hist[pb], m * (np - pr));
    }
    p.ws.nsplits[b] = count;
  }
  __syncthreads();
  if (tid == 0) {
    int pos = 0;
    for (int r = kSplitBlocks; r >= 1; --r) {
      bucket[r] = pos;
      pos += hist[r];
    }
    p.ws.header[kHdrTotal] = pos * p.num_kv_heads;
    p.ws.header[kHdrNext] = 0;
    p.ws.header[kHdrDone] = 0;
    p.ws.header[kHdrSignature] = p.signature;
  }
  __syncthreads();

  // pass 3: place every unit of a sequence, in block order, into its size's
  // bucket: (b, first block, split index << 16 | blocks, context length)
  for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
    int ctx = p.context_lens[b] - p.ctx_offset;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    int nsplit, base, big;
    split_shape((ctx + kBlockSize - 1) / kBlockSize, p.split_blocks, nsplit, base, big);
    int cut = cut_all;
    if (big * pieces_of(base + 1, cut, p.piece_blocks) + (nsplit - big) * pieces_of(base, cut, p.piece_blocks) > p.max_splits)
      cut = 0;
    // reserve this sequence's slots in each bucket it uses
    int at[2][2];  // [split size k][piece size pb + 1 / pb]
    for (int k = 0; k < 2; ++k) {
      const int n = base + 1 - k, m = k ? nsplit - big : big;
      at[k][0] = at[k][1] = 0;
      if (m == 0 || n == 0) continue;
      const int np = pieces_of(n, cut, p.piece_blocks);
      const int pb = n / np, pr = n - pb * np;
      if (pr) at[k][0] = atomicAdd(&bucket[pb + 1], m * pr);
      if (np - pr) at[k][1] = atomicAdd(&bucket[pb], m * (np - pr));
    }
    int first = 0, si = 0;
    for (int s = 0; s < nsplit; ++s) {
      const int k = s < big ? 0 : 1;
      const int n = base + 1 - k;
      const int np = pieces_of(n, cut, p.piece_blocks);
      const int pb = n / np, pr = n - pb * np;
      for (int j = 0; j < np; ++j) {
        const int sz = j < pr ? pb + 1 : pb;
        const int pos = j < pr ? at[k][0]++ : at[k][1]++;
        units[pos] = make_int4(b, first, (si << 16) | sz, ctx);
        first += sz;
        ++si;
      }
    }
  }
}

// ------------------------------------------------------------ grouped plan
// A grouped decode's batch is made of groups of consecutive sequences whose
// tables start with the same blocks (the branches of a forked prompt, the
// requests on one system prompt: "vLLM: treating the KV cache as virtual
// memory", section 碎片从哪里来, and the OS-lab appendix, section 4.3, where
// forked tables point at the same blocks).  The plan makes two kinds of
// unit: a shared unit covers a split of a group's shared blocks for up to
// `chunk` members at once (their m * G query rows read every block once),
// and an own unit a split of one sequence's blocks past the shared ones.  A
// sequence's splits are its group's shared splits (indices 0 ..) followed by
// its own; the attention launch merges them (a queue of ready merges that
// warps out of items take).
struct GroupArgs {
  const int32_t* group_start;   // [num_groups + 1], or null: one group of every sequence
  const int32_t* group_blocks;  // [num_groups] shared blocks, or null: single_blocks
  int num_groups;
  int single_blocks;
  int chunk;                    // most members of one shared unit
  int nwarps;                   // math warps of the attention launch
  int teams;                    // the attention launch can merge in teams (rings of >= 2 stages)
  int small;                    // the per-sequence and per-group arrays fit the plan's
                                //   shared memory (kGroupedPlanSmallSeqs; see grouped_plan_smem)
  int32_t* gp;                  // workspace [num_groups]: shared blocks that passed the checks
  int32_t* seq_prefix;          // workspace [num_seqs]: each sequence's shared blocks
  int32_t* seq_ctx;             // workspace [num_seqs]: context lengths, clamped
  int32_t* seq_group;           // workspace [num_seqs]: each sequence's group
  int2* seq_chunk;              // workspace [num_seqs]: its chunk's first member, members
  int4* chunk_plan;             // workspace [num_seqs]: at a chunk's first member, its cut
                                //   (absorbs, own blocks absorbed, shared splits, last shared)
};

__device__ __forceinline__ int group_of(const GroupArgs& ga, int b) {
  if (!ga.group_start) return 0;
  int lo = 0, hi = ga.num_groups - 1;  // the last g with group_start[g] <= b
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ga.group_start[mid] <= b) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// A chunk of at most kAbsorbMembers members whose blocks past the shared
// ones add up to at most kAbsorbBlocks takes them into its last shared unit:
// one unit then covers the chunk's last shared blocks (every row) and each
// member's own blocks (its rows only), so the members need no units of their
// own and all of them have the same splits.
constexpr int kAbsorbMembers = 4;
constexpr int kAbsorbBlocks = 16;
// flag in the blocks byte of a unit (blocks <= 32 use bits 0-5)
constexpr int kUnitOwn = 0x80;    // the unit also covers the members' own blocks
constexpr int kUnitBlocks = 0x3f;

struct ChunkPlan {
  bool absorb;
  int own;          // absorbed: the members' own blocks in all
  int ns;           // shared splits (absorbed: the last one carries the own blocks)
  int last_shared;  // absorbed: shared blocks of the last split
};

// Parts that `total` blocks are cut into for units of about sp (>= 16)
// blocks: rounded down, so that the units are no more than the math warps
// (one wave), and no part above 32 blocks.
__device__ __forceinline__ int shared_parts(int total, int sp) {
  int n = total / sp;
  const int at_most_32 = (total + kSplitBlocks - 1) / kSplitBlocks;
  if (n < at_most_32) n = at_most_32;
  return n < 1 ? 1 : n;
}

// Balanced parts: n parts of `total` blocks, the first `big` one larger.
__device__ __forceinline__ void parts_shape(int total, int n, int& base, int& big) {
  base = n ? total / n : 0;
  big = n ? total - base * n : 0;
}

// How the chunk of m members from b0, sharing P blocks, is cut (shared
// splits of about sp blocks).
__device__ __forceinline__ ChunkPlan plan_chunk(const GroupArgs& ga, int b0, int m, int P,
                                                int sp) {
  ChunkPlan c;
  c.absorb = false;
  c.own = 0;
  c.last_shared = 0;
  if (P > 0 && m <= kAbsorbMembers) {
    int own = 0;
    for (int i = 0; i < m; ++i) own += (ga.seq_ctx[b0 + i] + kBlockSize - 1) / kBlockSize - P;
    if (own <= kAbsorbBlocks) {
      const int total = P + own;
      int ns = shared_parts(total, sp);
      if (ns > P) ns = P;
      int last = P;
      if (ns <= 1) {
        ns = 1;
      } else {
        const int size = (total + ns - 1) / ns;
        last = size - own < 1 ? 1 : size - own;
        if (P - last < ns - 1) last = P - (ns - 1);
      }
      if (last + own <= kSplitBlocks) {
        c.absorb = true;
        c.own = own;
        c.ns = ns;
        c.last_shared = last;
      }
    }
  }
  if (!c.absorb) c.ns = shared_parts(P, sp);
  return c;
}

constexpr int kGroupedPlanThreads = 512;
// A batch of at most this many sequences and groups keeps the plan's
// per-sequence and per-group arrays in shared memory: every pass of the plan
// reads what the last one wrote, and from L2 those reads made the plan a
// chain of round trips (20 us per step on the 128-branch sampling batch).
constexpr int kGroupedPlanSmallSeqs = 1024;
inline size_t grouped_plan_smem(int num_seqs, int num_groups) {
  return size_t(num_seqs) * (16 + 8 + 3 * 4) + size_t(2 * num_groups + 1) * 4;
}

__global__ void __launch_bounds__(kGroupedPlanThreads) grouped_plan_kernel(const Params p,
                                                                           const GroupArgs gin) {
  constexpr int NT = kGroupedPlanThreads;
  __shared__ int hist[kSplitBlocks + 2];
  __shared__ int bucket[kSplitBlocks + 2];
  __shared__ int cut_s, bad_s, sp_s, merges_s, team_s, chunks_s, chunk_ctr;
  __shared__ unsigned long long work_s;
  extern __shared__ __align__(16) unsigned char plan_arrays[];
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();  // the previous kernel may still read the workspace
  const int tid = threadIdx.x;
  // the arrays the passes share: in shared memory for a small batch (the
  // run's seq_ctx and seq_prefix are copied out at the end), else in the
  // workspace
  GroupArgs ga = gin;
  if (gin.small) {
    const int B = p.num_seqs, G = gin.group_start ? gin.num_groups : 1;
    ga.chunk_plan = reinterpret_cast<int4*>(plan_arrays);
    ga.seq_chunk = reinterpret_cast<int2*>(ga.chunk_plan + B);
    ga.seq_ctx = reinterpret_cast<int32_t*>(ga.seq_chunk + B);
    ga.seq_group = ga.seq_ctx + B;
    ga.seq_prefix = ga.seq_group + B;
    ga.gp = ga.seq_prefix + B;
    if (gin.group_start) {
      int32_t* starts = ga.gp + G;
      for (int g = tid; g <= G; g += NT) starts[g] = gin.group_start[g];
      ga.group_start = starts;
    }
    __syncthreads();
  }
  const int ng = ga.group_start ? ga.num_groups : 1;
  const int cap = p.max_blocks * kBlockSize;
  const int mb = p.max_blocks;
  int4* units = reinterpret_cast<int4*>(p.ws.units);
  if (tid < kSplitBlocks + 2) hist[tid] = 0;
  if (tid == 0) {
    bad_s = ga.group_start && (ga.group_start[0] != 0 || ga.group_start[ng] != p.num_seqs);
    work_s = 0;
    merges_s = 0;
    team_s = 1;
    chunks_s = 0;
    chunk_ctr = 0;
  }
  __syncthreads();
  // group starts must not decrease (every thread checks its share)
  if (ga.group_start) {
    bool down = false;
    for (int g = tid; g < ng; g += NT) down |= ga.group_start[g] > ga.group_start[g + 1];
    if (down) bad_s = 1;
  }
  __syncthreads();
  // With unusable group arrays every sequence decodes on its own.
  const bool bad = bad_s;
  if (bad && tid == 0) dev::flag_status(p.status, kStatusBounds);
  for (int g = tid; g < ng; g += NT) {
    int nb = bad ? 0 : (ga.group_blocks ? ga.group_blocks[g] : ga.single_blocks);
    if (nb < 0 || nb > mb) {
      dev::flag_status(p.status, kStatusBounds);
      nb = 0;
    }
    ga.gp[g] = nb;
  }
  // every sequence's group and clamped context
  for (int b = tid; b < p.num_seqs; b += NT) {
    ga.seq_group[b] = bad ? 0 : group_of(ga, b);
    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > cap) {
      dev::flag_status(p.status, kStatusBounds);
      ctx = ctx < 0 ? 0 : cap;
    }
    ga.seq_ctx[b] = ctx;
    for (int h = 0; h < p.num_kv_heads; ++h) {
      p.ws.arrivals[size_t(b) * p.num_kv_heads + h] = 0;
      p.ws.mqueue[size_t(b) * p.num_kv_heads + h] = 0;
    }
  }
  __syncthreads();
  // Every member's context must cover the shared blocks and its table must
  // start with the first member's entries; a group with a member that does
  // not keeps no shared blocks (its members then decode on their own, which
  // gives the same attention).  The contexts one thread per sequence; the
  // tables eight entries per thread over all (member, entry) pairs, so that
  // every load is in flight at once.  A plan of one shared prefix gets no
  // tables (the run checks them).
  for (int b = tid; b < p.num_seqs && !bad; b += NT) {
    const int g = ga.seq_group[b];
    const int nb = ga.gp[g];
    const int ctx = p.context_lens[b];
    if (nb > 0 && (ctx < nb * kBlockSize || ctx > cap)) {
      atomicExch(&ga.gp[g], 0);
      dev::flag_status(p.status, kStatusBounds);
    }
  }
  if (!bad && p.block_tables) {
    const int per_seq = (mb + 7) / 8;
    const long long items = (long long)p.num_seqs * per_seq;
    for (long long i = tid; i < items; i += NT) {
      const int b = int(i / per_seq), j0 = int(i - (long long)b * per_seq) * 8;
      const int g = ga.seq_group[b];
      const int nb = ga.gp[g];
      const int first = ga.group_start ? ga.group_start[g] : 0;
      if (j0 >= nb || b == first) continue;
      const int32_t* row = p.block_tables + size_t(b) * mb;
      const int32_t* lead = p.block_tables + size_t(first) * mb;
      bool differ = false;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (j0 + k < nb) differ |= __ldg(row + j0 + k) != __ldg(lead + j0 + k);
      if (differ) {
        atomicExch(&ga.gp[g], 0);
        dev::flag_status(p.status, kStatusBounds);
      }
    }
  }
  __syncthreads();
  // per sequence: its shared blocks and chunk (first member, members); the
  // work (blocks per KV head) of the own blocks and of every chunk's shared
  // blocks, which sizes the shared splits (summed per thread, then per warp:
  // one 64-bit shared atomic per sequence, all on one word, took 6 us)
  unsigned long long work = 0;
  for (int b = tid; b < p.num_seqs; b += NT) {
    const int g = ga.seq_group[b];
    const int nb = bad ? 0 : ga.gp[g];
    const int first = ga.group_start && !bad ? ga.group_start[g] : 0;
    const int end = ga.group_start && !bad ? ga.group_start[g + 1] : p.num_seqs;
    const int b0 = first + (b - first) / ga.chunk * ga.chunk;
    const int m = end - b0 < ga.chunk ? end - b0 : ga.chunk;
    ga.seq_prefix[b] = nb;
    ga.seq_chunk[b] = make_int2(b0, m);
    unsigned long long w = (ga.seq_ctx[b] + kBlockSize - 1) / kBlockSize - nb;
    if (b == b0) w += nb;  // the chunk's shared blocks, read once
    work += w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) work += __shfl_down_sync(0xffffffffu, work, o);
  if ((tid & 31) == 0 && work) atomicAdd(&work_s, work);
  __syncthreads();
  if (tid == 0) {
    // shared splits of about the work one math warp gets, 16 to 32 blocks
    // (the workspace holds a sequence's splits for sizes of 16 and more)
    const unsigned long long per_warp =
        (work_s * p.num_kv_heads + ga.nwarps - 1) / (unsigned long long)ga.nwarps;
    sp_s = per_warp < kMinSplitBlocks ? kMinSplitBlocks
                                      : (per_warp > kSplitBlocks ? kSplitBlocks : int(per_warp));
  }
  __syncthreads();
  const int sp = sp_s;
  // every chunk's cut, once (by the thread of its first member)
  for (int b = tid; b < p.num_seqs; b += NT) {
    const int2 cm = ga.seq_chunk[b];
    const int P = ga.seq_prefix[b];
    if (b != cm.x || P == 0) continue;
    const ChunkPlan c = plan_chunk(ga, b, cm.y, P, sp);
    ga.chunk_plan[b] = make_int4(c.absorb, c.own, c.ns, c.last_shared);
  }
  __syncthreads();
  // Teams: when every sequence shares blocks with its chunk, every chunk
  // takes its members' own blocks into its last shared split (so no unit
  // covers one sequence alone) with at most kTeamWarps splits, and the
  // (chunk, KV head) pairs fit the launch's teams of kTeamWarps warps, the
  // splits of each pair go to one team of one CTA and are merged there, in
  // shared memory.
  for (int b = tid; b < p.num_seqs; b += NT) {
    const int2 cm = ga.seq_chunk[b];
    if (ga.seq_prefix[b] == 0) {
      team_s = 0;
      continue;
    }
    const int4 c = ga.chunk_plan[cm.x];
    if (!c.x || c.z > kTeamWarps) team_s = 0;
    if (b == cm.x) atomicAdd(&chunks_s, 1);
  }
  __syncthreads();
  const bool team = ga.teams && team_s && p.num_seqs > 0 &&
                    (long long)chunks_s * p.num_kv_heads * kTeamWarps <= ga.nwarps &&
                    (long long)chunks_s * kTeamWarps <= (long long)p.num_seqs * p.max_splits;
  // a sequence's own blocks that become units of its own (none when its
  // chunk absorbs them), and its chunk's shared splits
  auto own_and_shared = [&](int b, int& own, int& pn) {
    const int P = ga.seq_prefix[b];
    pn = 0;
    own = (ga.seq_ctx[b] + kBlockSize - 1) / kBlockSize - P;
    if (P > 0) {
      const int4 c = ga.chunk_plan[ga.seq_chunk[b].x];
      pn = c.z;
      if (c.x) own = 0;
    }
  };
  // shared units of the chunk whose first member is b: sizes into counts
  auto chunk_units = [&](int b, int* counts) {
    const int4 c = ga.chunk_plan[b];
    const int P = ga.seq_prefix[b];
    if (c.x) {
      // the shared blocks before the last split, in ns - 1 balanced parts
      const int k = c.z - 1, X = P - c.w;
      if (k > 0) {
        const int base = X / k, big = X % k;
        if (big) atomicAdd(&counts[base + 1], big);
        if (k - big) atomicAdd(&counts[base], k - big);
      }
      atomicAdd(&counts[c.w + c.y], 1);
    } else {
      int base, big;
      parts_shape(P, c.z, base, big);
      if (big) atomicAdd(&counts[base + 1], big);
      if (c.z - big) atomicAdd(&counts[base], c.z - big);
    }
  };

  // pass 1: unit sizes before any cut
  for (int b = tid; b < p.num_seqs; b += NT) {
    int own, pn;
    own_and_shared(b, own, pn);
    int nsplit, base, big;
    split_shape(own, p.split_blocks, nsplit, base, big);
    if (big) atomicAdd(&hist[base + 1], big);
    if (nsplit - big) atomicAdd(&hist[base], nsplit - big);
    if (b == ga.seq_chunk[b].x && ga.seq_prefix[b] > 0) chunk_units(b, hist);
  }
  __syncthreads();
  if (tid == 0) {
    // largest size `cut` such that all units of at most `cut` blocks hold no
    // more than the tail's share of the work (only own units are cut)
    const long long budget = p.tail_blocks / p.num_kv_heads;
    long long acc = 0;
    int cut = 0;
    while (cut < kSplitBlocks && acc + (long long)hist[cut + 1] * (cut + 1) <= budget) {
      ++cut;
      acc += (long long)hist[cut] * cut;
    }
    cut_s = cut;
  }
  __syncthreads();
  const int cut_all = cut_s;
  if (tid < kSplitBlocks + 2) hist[tid] = 0;
  __syncthreads();

  // pass 2: sizes of the final units, and every sequence's split count
  for (int b = tid; b < p.num_seqs; b += NT) {
    int own, pn;
    own_and_shared(b, own, pn);
    int nsplit, base, big;
    split_shape(own, p.split_blocks, nsplit, base, big);
    int cut = cut_all;
    if (pn + big * pieces_of(base + 1, cut, p.piece_blocks) +
            (nsplit - big) * pieces_of(base, cut, p.piece_blocks) > p.max_splits)
      cut = 0;
    int count = 0;
    for (int k = 0; k < 2; ++k) {  // the two split sizes
      const int n = base + 1 - k, mm = k ? nsplit - big : big;
      if (mm == 0 || n == 0) continue;
      const int np = pieces_of(n, cut, p.piece_blocks);
      count += mm * np;
      const int pb = n / np, pr = n - pb * np;
      if (pr) atomicAdd(&hist[pb + 1], mm * pr);
      if (np - pr) atomicAdd(&hist[pb], mm * (np - pr));
    }
    p.ws.nsplits[b] = pn + count;
    if (pn + count > 1) atomicAdd(&merges_s, 1);
    if (b == ga.seq_chunk[b].x && ga.seq_prefix[b] > 0) chunk_units(b, hist);
  }
  __syncthreads();
  if (tid == 0) {
    int pos = 0;
    for (int r = kSplitBlocks; r >= 1; --r) {
      bucket[r] = pos;
      pos += hist[r];
    }
    p.ws.header[kHdrTotal] = team ? chunks_s * p.num_kv_heads * kTeamWarps : pos * p.num_kv_heads;
    p.ws.header[kHdrNext] = 0;
    p.ws.header[kHdrDone] = 0;
    p.ws.header[kHdrQHead] = 0;
    p.ws.header[kHdrQTail] = 0;
    p.ws.header[kHdrQDone] = 0;
    p.ws.header[kHdrMerges] = team ? 0 : merges_s * p.num_kv_heads;
    p.ws.header[kHdrTeam] = team ? kTeamWarps : 0;
    p.ws.header[kHdrSignature] = p.signature;
  }
  __syncthreads();

  // pass 3: place the units.  Own units: (b, first block, split index << 16
  // | blocks, context), split indices after the chunk's shared ones.
  // Shared units: (first member, first block, split index << 16 | members
  // << 8 | kUnitOwn for a last split that absorbs | blocks, shared tokens).
  // With teams, chunk i's splits take places kTeamWarps i .. (the run reads
  // them once per KV head), unused places hold b = -1.
  for (int b = tid; b < p.num_seqs; b += NT) {
    int own, pn;
    own_and_shared(b, own, pn);
    const int P = ga.seq_prefix[b], ctx = ga.seq_ctx[b];
    int nsplit, base, big;
    split_shape(own, p.split_blocks, nsplit, base, big);
    int cut = cut_all;
    if (pn + big * pieces_of(base + 1, cut, p.piece_blocks) +
            (nsplit - big) * pieces_of(base, cut, p.piece_blocks) > p.max_splits)
      cut = 0;
    int at[2][2];
    for (int k = 0; k < 2; ++k) {
      const int n = base + 1 - k, mm = k ? nsplit - big : big;
      at[k][0] = at[k][1] = 0;
      if (mm == 0 || n == 0) continue;
      const int np = pieces_of(n, cut, p.piece_blocks);
      const int pb = n / np, pr = n - pb * np;
      if (pr) at[k][0] = atomicAdd(&bucket[pb + 1], mm * pr);
      if (np - pr) at[k][1] = atomicAdd(&bucket[pb], mm * (np - pr));
    }
    int first = P, si = pn;
    for (int s = 0; s < nsplit; ++s) {
      const int k = s < big ? 0 : 1;
      const int n = base + 1 - k;
      const int np = pieces_of(n, cut, p.piece_blocks);
      const int pb = n / np, pr = n - pb * np;
      for (int j = 0; j < np; ++j) {
        const int sz = j < pr ? pb + 1 : pb;
        const int pos = j < pr ? at[k][0]++ : at[k][1]++;
        units[pos] = make_int4(b, first, (si << 16) | sz, ctx);
        first += sz;
        ++si;
      }
    }
    const int2 cm = ga.seq_chunk[b];
    if (b != cm.x || P == 0) continue;
    // this thread places its chunk's shared units
    const int4 c = ga.chunk_plan[b];
    int sn, sbase, sbig;
    if (c.x) {
      sn = c.z - 1;  // the parts before the last split
      parts_shape(P - c.w, sn, sbase, sbig);
    } else {
      sn = c.z;
      parts_shape(P, sn, sbase, sbig);
    }
    const int place = team ? atomicAdd(&chunk_ctr, 1) * kTeamWarps : 0;
    int off = 0;
    for (int s = 0; s < sn; ++s) {
      const int sz = s < sbig ? sbase + 1 : sbase;
      const int pos = team ? place + s : atomicAdd(&bucket[sz], 1);
      units[pos] = make_int4(b, off, (s << 16) | (cm.y << 8) | sz, P * kBlockSize);
      off += sz;
    }
    if (c.x) {
      const int pos = team ? place + c.z - 1 : atomicAdd(&bucket[c.w + c.y], 1);
      units[pos] = make_int4(b, off, ((c.z - 1) << 16) | (cm.y << 8) | kUnitOwn | c.w,
                             P * kBlockSize);
    }
    if (team)
      for (int s = c.z; s < kTeamWarps; ++s) units[place + s] = make_int4(-1, 0, 0, 0);
  }
  if (gin.small) {
    // what the run reads: the clamped contexts and every sequence's shared blocks
    for (int b = tid; b < p.num_seqs; b += NT) {
      gin.seq_ctx[b] = ga.seq_ctx[b];
      gin.seq_prefix[b] = ga.seq_prefix[b];
    }
  }
}

// --------------------------------------------------------- tensor-core path
// Merges the nsplit partial results (o, lse) of the query heads of (b, g)
// into out: out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M), M the largest
// lse_s (a log-sum-exp merge; the partial o_s are already normalised).  One
// warp does it, latency-bound on L2 reads of data other SMs just wrote (hence
// .cg loads), so the reads are batched into as few rounds as the registers
// allow: lane l owns the float4 columns c = l + 32 k (k < NK) of the group's
// G x D outputs and loads, for U splits at once, their o_s columns and the
// lse_s of each column's head; the running largest lse of each column is
// carried across rounds (the sums are rescaled when it grows), so no round
// waits for another's results.
// Where the partial results of one (b, g) live and where its merge goes.
struct MergeArgs {
  const float* lse;   // part_lse at (b, split 0, head g G); split stride Hq
  const float4* po;   // part_o at the same row, as float4
  void* out;          // out row of head g G of sequence b
  float* cas_o;       // suffix mode: fp32 o rows of head g G (else null)
  float* cas_lse;     // suffix mode: base-2 log-sum-exp of head g G
  int G, Hq, nsplit;
};

template <typename T, int D, int NK, int L>
__device__ __forceinline__ void merge_splits(const MergeArgs a, int lane) {
  using M = dev::Mma<T>;
  constexpr int U = NK == 1 ? 16 : (L / NK > 0 ? L / NK : 1);  // splits per round
  const int G = a.G, Hq = a.Hq, nsplit = a.nsplit;
  const int C = G * D / 4;  // float4 columns of the group's outputs
  const float* lse = a.lse;
  const float4* po = a.po;
  const size_t split4 = size_t(Hq) * D / 4;  // float4s between two splits

  // per column k of this lane: the largest lse so far, and the sums of
  // 2^(lse_s - largest) o_s and of 2^(lse_s - largest)
  float mx[NK], sum[NK];
  float4 acc[NK];
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    mx[k] = -INFINITY;
    sum[k] = 0.f;
    acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int sp0 = 0; sp0 < nsplit; sp0 += U) {
    float4 v[U][NK];
    float w[U][NK];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int k = 0; k < NK; ++k) {
        const int sp = sp0 + u, c = lane + 32 * k;
        const bool on = sp < nsplit && c < C;
        v[u][k] = on ? __ldcg(po + size_t(sp) * split4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        w[u][k] = on ? __ldcg(lse + size_t(sp) * Hq + (4 * c) / D) : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int k = 0; k < NK; ++k) {
        if (w[u][k] == -INFINITY) continue;  // weight 0 (also: nothing to load)
        const float mn = fmaxf(mx[k], w[u][k]);
        const float r = dev::fast_exp2(mx[k] - mn);  // 0 while mx is -inf
        const float e = dev::fast_exp2(w[u][k] - mn);
        mx[k] = mn;
        sum[k] = sum[k] * r + e;
        acc[k].x = acc[k].x * r + e * v[u][k].x;
        acc[k].y = acc[k].y * r + e * v[u][k].y;
        acc[k].z = acc[k].z * r + e * v[u][k].z;
        acc[k].w = acc[k].w * r + e * v[u][k].w;
      }
    }
  }
  T* orow = static_cast<T*>(a.out);
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    const int c = lane + 32 * k;
    if (c < C) {
      const float inv = 1.f / sum[k];
      if (a.cas_o) {
        *reinterpret_cast<float4*>(a.cas_o + 4 * c) =
            make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
      } else {
        uint2 pk;
        pk.x = M::pack(acc[k].x * inv, acc[k].y * inv);
        pk.y = M::pack(acc[k].z * inv, acc[k].w * inv);
        *reinterpret_cast<uint2*>(orow + 4 * c) = pk;
      }
      // the lse of a head, from the lane holding its first column
      if (a.cas_lse && (4 * c) % D == 0) a.cas_lse[(4 * c) / D] = mx[k] + log2f(sum[k]);
    }
  }
}

// L: float4 loads in flight per lane (24 measured 1 % faster than 16 for the
// MHA and GQA decode on GB300).
template <typename T, int D, int L>
__device__ __forceinline__ void merge_dispatch(const MergeArgs a, int lane) {
  const int nk = (a.G * D / 4 + 31) / 32;
  switch (nk) {
    case 1: merge_splits<T, D, 1, L>(a, lane); break;
    case 2: merge_splits<T, D, 2, L>(a, lane); break;
    case 3: merge_splits<T, D, 3, L>(a, lane); break;
    case 4: merge_splits<T, D, 4, L>(a, lane); break;
    default:
      if constexpr (D == 128) {
        switch (nk) {
          case 5: merge_splits<T, D, 5, L>(a, lane); break;
          case 6: merge_splits<T, D, 6, L>(a, lane); break;
          case 7: merge_splits<T, D, 7, L>(a, lane); break;
          default: merge_splits<T, D, 8, L>(a, lane); break;
        }
      }
  }
}

// Floats between two rows of a split's results in a team warp's ring (16
// bytes of padding, so the four rows a store instruction writes fall in
// different banks); the 16 rows' base-2 lse follow the rows.
template <int D>
constexpr int team_row() { return D + 4; }

// A team's merge: member rows r0 .. r0 + G - 1 of the ns splits whose results
// (o normalised, fp32, then the rows' lse) sit in the rings of the team's
// warps, ring_bytes apart from ring0, merged with log-sum-exp weights into
// out (the member's G x D outputs).  Lane l owns the float4 columns l + 32 k.
template <typename T, int D>
__device__ __forceinline__ void team_merge(const uint8_t* ring0, size_t ring_bytes, int ns,
                                           int r0, int G, T* out, int lane) {
  using M = dev::Mma<T>;
  constexpr int RS = team_row<D>();
  const int C = G * D / 4;
  for (int c = lane; c < C; c += 32) {
    const int r = r0 + (4 * c) / D, d = (4 * c) % D;
    float l[kTeamWarps];
    float mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < kTeamWarps; ++s) {
      l[s] = s < ns ? reinterpret_cast<const float*>(ring0 + s * ring_bytes)[16 * RS + r]
                    : -INFINITY;
      mx = fmaxf(mx, l[s]);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sum = 0.f;
#pragma unroll
    for (int s = 0; s < kTeamWarps; ++s) {
      if (s < ns) {
        const float w = dev::fast_exp2(l[s] - mx);
        const float4 v = *reinterpret_cast<const float4*>(
            reinterpret_cast<const float*>(ring0 + s * ring_bytes) + r * RS + d);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
        sum += w;
      }
    }
    const float inv = 1.f / sum;
    uint2 pk;
    pk.x = M::pack(acc.x * inv, acc.y * inv);
    pk.y = M::pack(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out + 4 * c) = pk;
  }
}

// A work item as a math warp holds it: registers only.  Lane j keeps the
// physical block of the item's logical block j (an item has at most 32).
// An item of a grouped decode may cover a block range that several
// consecutive sequences share (the m members b .. b + m - 1 of a group,
// m * G query rows); otherwise it is one sequence's (m = 1, G rows).
struct Item {
  int b;  // sequence (first member), or -1 once the work list is exhausted
  int g, s, nblk, first, ctx, nsplit;
  int m, rows;  // members and query rows
  int flags;    // kUnitOwn of the unit
  int phys;
  // kUnitOwn items, lane j for block j: the member the block belongs to (-1:
  // shared by all rows), its tokens in context, and the row of the member's
  // new token in it (-1: none); lane i < m: member i's new-token slot
  int bmem, bvalid, bpatch;
  long long mslot;
  unsigned okmask;  // members whose new token is stored and attended
  int slot;  // fused append: the new token's slot, or -1 (none / not this item)
  bool patch;  // the new token is this item's last attended token
};

// NT: query-row tiles of 8 per item (1: up to 8 rows, one sequence's query
// group; 2: up to 16, the rows of the members of a group sharing the item's
// blocks).
template <typename T, int D, int W, int NT>
__global__ void __launch_bounds__(W * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  using S = Smem<D, W, NT>;
  using M = dev::Mma<T>;
  constexpr int KT = D / 16;      // 16-wide steps along head_dim
  constexpr int kTeamRow = team_row<D>();
  static_assert(NT == 1 || (W % kTeamWarps == 0 &&
                            (16 * kTeamRow + 16) * 4 <= 2 * S::kStageBytes),
                "a team warp's results fit the first two stages of its ring");
  constexpr int HALVES = D / 64;  // 128-byte TMA boxes per tile row
  // The next item is claimed when this many blocks of the current one are
  // still to be issued: its claim takes one pipeline step per block (counter,
  // unit, table entries, query copy), so it is ready when the ring wants it.
  constexpr int kLead = 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int G = p.group;
  // the member of each of this lane's two query columns, per row tile
  // (computed once: the divisions in the block loop cost the grouped decode
  // 1.6 us per layer)
  int mc0[NT], mc1[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int qr = 8 * t + 2 * ((threadIdx.x & 31) & 3);
    mc0[t] = qr / G;
    mc1[t] = (qr + 1) / G;
  }
  const int NS = p.stages;  // ring stages of each warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + size_t(warp) * NS * S::kStageBytes;
  uint16_t* qbuf = reinterpret_cast<uint16_t*>(smem + size_t(W) * NS * S::kStageBytes +
                                               size_t(warp) * S::kQBytes);
  uint64_t* my_full = reinterpret_cast<uint64_t*>(smem + size_t(W) * NS * S::kStageBytes +
                                                  size_t(W) * S::kQBytes) +
                      warp * (kWarpStages + 1);
  uint64_t* my_q = my_full + kWarpStages;
  // grouped decode in teams: one barrier per team of kTeamWarps warps
  uint64_t* team_bars = reinterpret_cast<uint64_t*>(smem + size_t(W) * NS * S::kStageBytes +
                                                    size_t(W) * S::kQBytes) +
                        W * (kWarpStages + 1);

  // Every warp owns its barriers, so no CTA-wide synchronisation is needed.
  if (lane == 0) {
    for (int i = 0; i < kWarpStages; ++i) dev::mbar_init(&my_full[i], 1);
    dev::mbar_init(my_q, 1);
    dev::mbar_fence_init();
    dev::prefetch_tensormap(&tmap_k);
    dev::prefetch_tensormap(&tmap_v);
  }
  __syncwarp();
  if constexpr (NT == 2) {
    // the team barriers are the CTA's: initialised before any warp goes on
    if (threadIdx.x == 0) {
      for (int i = 0; i < W / kTeamWarps; ++i) dev::mbar_init(&team_bars[i], kTeamWarps);
      dev::mbar_fence_init();
    }
    __syncthreads();
  }
  // The next kernel of the stream may start launching; it waits for this
  // one's completion before it touches memory.
  dev::grid_launch_dependents();
  // This warp's first item, dealt statically.  W consecutive items (the
  // heads of one unit, reading neighbouring tiles) per CTA measured best
  // when every warp gets one (MHA 7B decode 0.868 of the measured copy
  // bandwidth dealt round robin, 0.883 so); a shorter list (a grouped decode
  // has at most one unit per warp) goes round robin over the SMs, or the
  // last SMs would idle (grouped decode 0.5-0.7 us faster per layer).
  // With teams (tm: a grouped plan that placed each (chunk, KV head)'s
  // splits as kTeamWarps consecutive items), team t goes to CTA t % (CTAs),
  // whose warps w with w / kTeamWarps == t / (CTAs) take its items.
  auto first_item = [&](int items, bool tm) {
    if constexpr (NT == 2) {
      if (tm)
        return ((warp / kTeamWarps) * int(gridDim.x) + int(blockIdx.x)) * kTeamWarps +
               warp % kTeamWarps;
    }
    return items < int(gridDim.x) * W ? warp * int(gridDim.x) + int(blockIdx.x)
                                      : int(blockIdx.x) * W + warp;
  };
  // item x -> its unit and KV head: the heads of a unit are consecutive
  // items, or (teams) the splits of a (chunk, head) are
  auto unit_of = [&](int x, bool tm, int& hg) {
    if constexpr (NT == 2) {
      if (tm) {
        const int t = x / kTeamWarps;
        hg = t % p.num_kv_heads;
        return (t / p.num_kv_heads) * kTeamWarps + x % kTeamWarps;
      }
    }
    hg = x % p.num_kv_heads;
    return x / p.num_kv_heads;
  };
  // While the kernel before this one finishes: warm L2 with the first blocks
  // of this warp's statically dealt first item.  The work list and tables may
  // still be changing (the previous kernel may be the plan), so this is only
  // a hint: every value is range-checked before it becomes an address, and
  // the real claim reads them again after the wait below.  How far: the
  // first 8 blocks when each query row has a KV head of its own (MHA: short
  // launches, whose start weighs most; 0.872 -> 0.882 of the measured copy
  // bandwidth per layer step on GB300), else 4 (GQA got 0.6 % slower with 8).
  {
    const long long cap = (long long)p.num_seqs * p.max_splits * p.num_kv_heads;  // items
    const int total0 = *reinterpret_cast<volatile int*>(&p.ws.header[kHdrTotal]);
    bool team0 = false;
    if constexpr (NT == 2)
      team0 = *reinterpret_cast<volatile int*>(&p.ws.header[kHdrTeam]) == kTeamWarps;
    const int x0 = first_item(total0, team0);
    int hg = 0;
    const int u0 = unit_of(x0, team0, hg);
    if (x0 < total0 && x0 < cap && u0 < (long long)p.num_seqs * p.max_splits) {
      // (read through L2 only: a line left in L1 now could be stale for the
      // claim's read of the same unit after the wait)
      const int4 u = __ldcg(reinterpret_cast<const int4*>(p.ws.units) + u0);
      const int n = u.z & kUnitBlocks;
      const int kWarmBlocks = p.group == 1 ? 8 : 4;
      if (u.x >= 0 && u.x < p.num_seqs && u.y >= 0 && n >= 1 && n <= kSplitBlocks &&
          p.table_offset + u.y + n <= p.max_blocks) {
        const int nb = n < kWarmBlocks ? n : kWarmBlocks;
        int phys = -1;
        if (lane < nb)
          phys = __ldcg(p.block_tables + size_t(u.x) * p.max_blocks + p.table_offset + u.y +
                        lane);
        for (int j = 0; j < nb; ++j) {
          const int pj = __shfl_sync(0xffffffffu, phys, j);
          if (pj < 0 || pj >= p.num_blocks) continue;
          // a (block, head) tile is 16 * D * 2 bytes: D / 4 lines of 128 bytes
          const size_t tile = (size_t(pj) * p.num_kv_heads + hg) * kBlockSize * D * 2;
          for (int l = lane; l < D / 4; l += 32) {
            dev::prefetch_l2(static_cast<const uint8_t*>(p.k_cache) + tile + size_t(l) * 128);
            dev::prefetch_l2(static_cast<const uint8_t*>(p.v_cache) + tile + size_t(l) * 128);
          }
        }
      }
    }
  }
  dev::grid_dependency_wait();  // the kernel before this one has completed
  TIME_MARK(0, dev::global_timer_ns());

  const unsigned long long tmo = p.timeout_ns;
  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  const int nwarps = int(gridDim.x) * W;
  const bool signed_ok =
      *reinterpret_cast<volatile int*>(&p.ws.header[kHdrSignature]) == p.signature;
  if (!signed_ok && blockIdx.x == 0 && threadIdx.x == 0) dev::flag_status(p.status, kStatusPlan);
  // a grouped decode placed in teams: the plan made sure that the teams fit
  // the launch and that the rings hold a split's results
  bool team = false, team_bad = false;
  if constexpr (NT == 2) {
    team = signed_ok &&
           *reinterpret_cast<volatile int*>(&p.ws.header[kHdrTeam]) == kTeamWarps;
    team_bad = team && (*reinterpret_cast<volatile int*>(&p.ws.header[kHdrTotal]) > nwarps ||
                        size_t(NS) * S::kStageBytes < size_t(16 * kTeamRow + 16) * 4);
    if (team_bad && blockIdx.x == 0 && threadIdx.x == 0) dev::flag_status(p.status, kStatusBounds);
  }
  const bool planned = signed_ok && !team_bad;
  const int total = planned ? *reinterpret_cast<volatile int*>(&p.ws.header[kHdrTotal]) : 0;
  const int4* units = reinterpret_cast<const int4*>(p.ws.units);

  const bool fused = p.slot_mapping != nullptr;
  const long long num_slots = (long long)p.num_blocks * kBlockSize;
  if (planned && warp == W - 1 && p.verify_prefix) {
    // one shared prefix: every table must start with sequence 0's entries
    const long long pairs = (long long)p.num_seqs * p.max_blocks;
    for (long long i = blockIdx.x * 32 + lane; i < pairs; i += gridDim.x * 32) {
      const int b = int(i / p.max_blocks), j = int(i % p.max_blocks);
      if (j < p.seq_prefix[b] && p.block_tables[i] != p.block_tables[j])
        dev::flag_status(p.status, kStatusBounds);
    }
  }
  if (planned && warp == W - 1) {
    // rows of empty sequences are zero; a new token of such a sequence is
    // still stored (it attends nothing)
    for (int b = blockIdx.x * 32 + lane; b < p.num_seqs; b += gridDim.x * 32) {
      if (p.cas_o && p.context_lens[b] - p.ctx_offset <= 0) {
        // suffix mode: nothing past the shared prefix (weight 0 in the merge).
        // A new token would then sit inside the shared blocks, which a
        // sequence never writes (copy-on-write gives it its own block first).
        for (int i = 0; i < Hq * D; ++i) p.cas_o[size_t(b) * Hq * D + i] = 0.f;
        for (int h = 0; h < Hq; ++h) p.cas_lse[size_t(b) * Hq + h] = -INFINITY;
        if (fused && p.slot_mapping[b] >= 0) dev::flag_status(p.status, kStatusBounds);
      } else if (p.seq_prefix && fused && p.context_lens[b] > 0 &&
                 p.context_lens[b] <= p.seq_prefix[b] * kBlockSize && p.slot_mapping[b] >= 0) {
        // grouped mode: the new token would sit inside the shared blocks,
        // which a sequence never writes; it is neither stored nor attended
        dev::flag_status(p.status, kStatusBounds);
      } else if (!p.cas_o && p.context_lens[b] <= 0) {
        uint4* row = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + size_t(b) * Hq * D);
        for (int i = 0; i < Hq * D * 2 / 16; ++i) row[i] = make_uint4(0, 0, 0, 0);
        const long long slot = fused ? p.slot_mapping[b] : -1;
        if (slot >= num_slots) dev::flag_status(p.status, kStatusBounds);
        if (slot >= 0 && slot < num_slots) {
          for (int h = 0; h < Hkv; ++h) {
            const size_t src = (size_t(b) * Hkv + h) * D / 8;
            const size_t dst = ((size_t(slot / kBlockSize) * Hkv + h) * kBlockSize +
                                size_t(slot % kBlockSize)) * D / 8;
            for (int c = 0; c < D / 8; ++c) {
              static_cast<uint4*>(const_cast<void*>(p.k_cache))[dst + c] =
                  static_cast<const uint4*>(p.k_new)[src + c];
              static_cast<uint4*>(const_cast<void*>(p.v_cache))[dst + c] =
                  static_cast<const uint4*>(p.v_new)[src + c];
            }
          }
        }
      }
    }
  }

  // ---- claim pipeline for the next item (one step per call of advance())
  //   1: the work counter's reply is awaited    2: the unit is being read
  //   3: the table entries are being read       4: `nxt` is complete
  Item cur, nxt;
  cur.b = nxt.b = -1;
  cur.g = cur.s = cur.nblk = cur.first = cur.ctx = cur.nsplit = cur.phys = 0;
  nxt.g = nxt.s = nxt.nblk = nxt.first = nxt.ctx = nxt.nsplit = nxt.phys = 0;
  cur.m = nxt.m = 1;
  cur.rows = nxt.rows = G;
  cur.flags = nxt.flags = 0;
  cur.bmem = nxt.bmem = -1;
  cur.bvalid = nxt.bvalid = 0;
  cur.bpatch = nxt.bpatch = -1;
  cur.mslot = nxt.mslot = -1;
  cur.okmask = nxt.okmask = 0u;
  int octx = 0;  // kUnitOwn claim: lane i < m holds member i's context
  cur.slot = nxt.slot = -1;
  cur.patch = nxt.patch = false;
  long long cslot = -1;  // slot_mapping[b] of the item being claimed
  int cstage = 1;
  // blocks of `nxt` whose physical block is known before its claim is
  // complete (a shared unit's shared blocks, from its stage 5 on), so that
  // their copies may start early
  int nxt_known = 0;
  int cx = first_item(total, team);  // first item of every warp: dealt statically
  int4 cu = make_int4(0, 0, 0, 0);
  int q_issued = 0, q_taken = 0;  // query copies issued into / read from qbuf
  auto finished = [&]() {
    // This warp takes no more items.  The last warp to get here returns the
    // counters to zero, so the next run on this plan starts clean.
    if (lane == 0 && planned) {
      __threadfence();
      if (atomicAdd(&p.ws.header[kHdrDone], 1) == nwarps - 1) {
        atomicExch(&p.ws.header[kHdrNext], 0);
        atomicExch(&p.ws.header[kHdrDone], 0);
      }
    }
  };
  auto advance = [&]() {
    if (cstage == 1) {
      const int x = __shfl_sync(0xffffffffu, cx, 0);
      if (x >= total) {
        nxt.b = -1;
        nxt.nblk = 0;
        cstage = 4;
        finished();
      } else {
        if constexpr (NT == 2) {
          int hg;
          cu = __ldg(&units[unit_of(x, team, hg)]);
          nxt.g = hg;
        } else {
          cu = __ldg(&units[x / Hkv]);
          nxt.g = x % Hkv;
        }
        cstage = 2;
      }
    } else if (cstage == 2) {
      if (NT == 2 && team && cu.x < 0) {
        // an unused place of a team: this warp takes no item
        nxt.b = -1;
        nxt.nblk = 0;
        cstage = 4;
        finished();
        return;
      }
      nxt.b = cu.x;
      nxt.first = cu.y;
      nxt.s = cu.z >> 16;
      nxt.m = (cu.z >> 8) & 0xff;
      nxt.nblk = cu.z & kUnitBlocks;
      nxt.flags = cu.z & kUnitOwn;
      nxt.ctx = cu.w;
      // a unit shared by several members (grouped plans only)
      if (nxt.m < 1 || NT == 1 || nxt.m * G > 8 * NT || nxt.b + nxt.m > p.num_seqs) {
        if (nxt.m != 0 || nxt.flags) dev::flag_status(p.status, kStatusBounds);
        nxt.m = 1;
        nxt.flags = 0;
      }
      if ((nxt.flags & kUnitOwn) && nxt.m > kAbsorbMembers) {
        dev::flag_status(p.status, kStatusBounds);
        nxt.flags &= ~kUnitOwn;
      }
      nxt.rows = nxt.m * G;
      nxt.nsplit = __ldg(&p.ws.nsplits[nxt.b]);
      // only an item of one sequence carries its new token
      cslot = fused && (cu.z & 0xff00) == 0 ? __ldg(&p.slot_mapping[nxt.b]) : -1;
      nxt.phys = lane < nxt.nblk
                     ? __ldg(&p.block_tables[size_t(nxt.b) * p.max_blocks + p.table_offset +
                                             nxt.first + lane])
                     : 0;
      nxt.bmem = -1;
      nxt.bvalid = nxt.ctx - (nxt.first + lane) * kBlockSize;
      nxt.bpatch = -1;
      nxt.okmask = 0u;
      nxt.mslot = -1;
      if (nxt.flags & kUnitOwn) {
        // the members' contexts and new-token slots, for the next step
        octx = lane < nxt.m ? __ldg(&p.context_lens[nxt.b + lane]) : 0;
        nxt.mslot = fused && lane < nxt.m ? __ldg(&p.slot_mapping[nxt.b + lane]) : -1;
        cstage = 5;
      } else {
        cstage = 3;
      }
    } else if (cstage == 5) {
      // kUnitOwn: after the shared blocks (they end at the group's shared
      // count P), member i's own blocks P .. ceil(ctx_i / 16) - 1, member
      // after member; lane j takes block j of that list
      nxt_known = nxt.nblk;  // the shared blocks' entries came with the unit
      const int P = nxt.first + nxt.nblk;
      const int own = lane < nxt.m ? max(0, (octx + kBlockSize - 1) / kBlockSize - P) : 0;
      int off = own;  // inclusive sum over lanes 0 .. lane
#pragma unroll
      for (int d = 1; d < kAbsorbMembers; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, off, d);
        if (lane >= d) off += v;
      }
      const int total = __shfl_sync(0xffffffffu, off, kAbsorbMembers - 1);
      off -= own;  // exclusive
      const int n0 = nxt.nblk;
      const int jj = lane - n0;
      int mem = -1, mctx = 0, moff = 0;
#pragma unroll
      for (int i = 0; i < kAbsorbMembers; ++i) {
        const int oi = __shfl_sync(0xffffffffu, off, i), ni = __shfl_sync(0xffffffffu, own, i);
        const int ci = __shfl_sync(0xffffffffu, octx, i);
        if (i < nxt.m && jj >= oi && jj < oi + ni) {
          mem = i;
          mctx = ci;
          moff = oi;
        }
      }
      if (n0 + total > kSplitBlocks) {  // the plan keeps every item within 32 blocks
        dev::flag_status(p.status, kStatusBounds);
        mem = -1;
      } else {
        nxt.nblk = n0 + total;
      }
      if (mem >= 0) {
        const int local = P + jj - moff;
        nxt.phys = __ldg(&p.block_tables[size_t(nxt.b + mem) * p.max_blocks + local]);
        nxt.bmem = mem;
        nxt.bvalid = mctx - local * kBlockSize;
        nxt.bpatch = local == (mctx + kBlockSize - 1) / kBlockSize - 1 ? (mctx - 1) % kBlockSize : -1;
      }
      cstage = 3;
    } else if (cstage == 3) {
      if (lane < nxt.nblk && (nxt.phys < 0 || nxt.phys >= p.num_blocks)) {
        dev::flag_status(p.status, kStatusBounds);
        nxt.phys = 0;
      }
      if (nxt.flags & kUnitOwn) {
        // the lane of a member's last block checks that member's new-token
        // slot against the position of its last token
        const long long ms = __shfl_sync(0xffffffffu, nxt.mslot, nxt.bmem < 0 ? 0 : nxt.bmem);
        bool ok = false;
        if (lane < nxt.nblk && nxt.bpatch >= 0 && ms >= 0) {
          ok = ms < num_slots && (long long)nxt.phys * kBlockSize + nxt.bpatch == ms;
          if (!ok) dev::flag_status(p.status, kStatusBounds);
        }
        if (!ok) nxt.bpatch = -1;
        nxt.okmask = __reduce_or_sync(0xffffffffu, ok ? 1u << nxt.bmem : 0u);
      }
      // Fused append: the item holding the sequence's last block stores the
      // new token's K/V row of its KV head and uses it as its last token.
      nxt.slot = -1;
      nxt.patch = false;
      if (fused && nxt.s == nxt.nsplit - 1 && cslot >= 0) {
        if (cslot >= num_slots) {
          dev::flag_status(p.status, kStatusBounds);
        } else {
          nxt.slot = int(cslot);
          const int last_phys = __shfl_sync(0xffffffffu, nxt.phys, nxt.nblk - 1);
          const long long at = (long long)last_phys * kBlockSize + (nxt.ctx - 1) % kBlockSize;
          nxt.patch = at == cslot;
          // a slot that is not the position of the sequence's last token
          if (!nxt.patch) dev::flag_status(p.status, kStatusBounds);
        }
      }
      // the G query rows of (b, g) (and the new K/V row) go to this warp's
      // staging buffer, which the current item no longer reads: its rows are
      // in registers
      const uint32_t rbytes = nxt.slot >= 0 ? 2u * D * 2 : 0u;
      if (lane == 0) dev::mbar_arrive_expect_tx(my_q, uint32_t(nxt.rows) * D * 2 + rbytes);
      __syncwarp();
      // lane r copies query row r (member r / G, head r % G of the group)
      // into row r of the buffer
      if (lane < nxt.rows)
        dev::bulk_load(qbuf + lane * S::kQRow,
                       static_cast<const uint8_t*>(p.q) +
                           ((size_t(nxt.b) + lane / G) * Hq + size_t(nxt.g) * G + lane % G) *
                               D * 2,
                       D * 2, my_q);
      if (rbytes && lane == 0) {
        const size_t row = (size_t(nxt.b) * Hkv + nxt.g) * D * 2;
        dev::bulk_load(qbuf + 8 * S::kQRow, static_cast<const uint8_t*>(p.k_new) + row, D * 2,
                       my_q);
        dev::bulk_load(qbuf + 8 * S::kQRow + D, static_cast<const uint8_t*>(p.v_new) + row, D * 2,
                       my_q);
      }
      ++q_issued;
      cstage = 4;
    }
  };
  auto request = [&]() {  // starts the claim of the next item
    if (lane == 0) cx = nwarps + atomicAdd(&p.ws.header[kHdrNext], 1);
    cstage = 1;
    nxt_known = 0;
  };

  // ---- issue cursor: blocks of `cur`, then of `nxt` once it is complete
  int cur_issued = 0, nxt_issued = 0;
  int ik = 0;   // blocks issued into the ring so far
  int ist = 0;  // ik % NS (kept as a count: NS is a launch value)
  const uint64_t policy = dev::l2_policy_evict_first();
  auto top_up = [&](int kc) {
    while (ik < kc + NS) {
      bool from_cur = cur_issued < cur.nblk;
      if (!from_cur && !(nxt_issued < (cstage == 4 ? nxt.nblk : nxt_known))) break;
      const int j = from_cur ? cur_issued++ : nxt_issued++;
      const int phys = __shfl_sync(0xffffffffu, from_cur ? cur.phys : nxt.phys, j);
      const int gg = from_cur ? cur.g : nxt.g;
      const int st = ist;
      if (++ist == NS) ist = 0;
      if (lane == 0) dev::mbar_arrive_expect_tx(&my_full[st], S::kStageBytes);
      __syncwarp();
      // lanes 0..HALVES-1 each issue one 128-byte-wide box of the K tile,
      // then of the V tile (one tensor map per instruction)
      if (lane < HALVES) {
        uint8_t* dst = ring + size_t(st) * S::kStageBytes + lane * 2048;
        const int y = (phys * Hkv + gg) * kBlockSize;
        dev::tma_load_2d(dst, &tmap_k, lane * 64, y, &my_full[st], policy);
        dev::tma_load_2d(dst + S::kTileBytes, &tmap_v, lane * 64, y, &my_full[st], policy);
      }
      ++ik;
    }
  };
  int kc = 0;            // blocks consumed so far
  int cst = 0, cph = 0;  // kc % NS and (kc / NS) & 1: the stage and phase to wait for
  // On a timeout: let this warp's copies in flight land, then give up.
  auto drain = [&]() {
    if (lane == 0) {
      for (int k = kc; k < ik; ++k)
        mbar_wait_bounded(&my_full[k % NS], (k / NS) & 1, tmo, p.status);
      if (q_issued > q_taken) mbar_wait_bounded(my_q, q_taken & 1, tmo, p.status);
    }
    __syncwarp();
  };

  // the first item, claimed in full before anything else (its blocks'
  // copies start as soon as their entries are known)
  while (cstage != 4) {
    advance();
    top_up(kc);
  }
#ifdef PA_PROFILE_TIMES
  int n_items = 0;
#endif
  for (;;) {
    // ---- move on to the next item
    cur = nxt;
    cur_issued = nxt_issued;
    nxt_issued = 0;
    nxt.b = -1;
    nxt.nblk = 0;
    cstage = 0;
    if (cur.b < 0) break;
    nxt_known = 0;
#ifdef PA_PROFILE_TIMES
    const unsigned long long item_t0 = dev::global_timer_ns();
#endif
    const int b = cur.b, g = cur.g, s = cur.s, ctx = cur.ctx, nblk = cur.nblk, first = cur.first;
    const int nsplit = cur.nsplit, rows = cur.rows;
    // the second row tile holds rows (warp-uniform)
    const bool two = NT == 2 && rows > 8;
    // B fragments of Q^T (k = head_dim, n = query head of the group)
    if (!mbar_wait_bounded(my_q, q_taken & 1, tmo, p.status)) {
      drain();
      return;
    }
    ++q_taken;
#ifdef PA_PROFILE_TIMES
    const unsigned long long qwait_ns = dev::global_timer_ns() - item_t0;
    unsigned long long merge_ns = 0;
#endif
    uint32_t qb0[NT][KT], qb1[NT][KT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int hq = 8 * t + (lane >> 2);
      const int n0 = 2 * (lane & 3);
      const uint16_t* qrow = qbuf + hq * S::kQRow + n0;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        qb0[t][kk] = hq < rows ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk) : 0u;
        qb1[t][kk] = hq < rows ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8) : 0u;
      }
    }
    // fused append: lane l < D/4 holds 16 bytes of the new K row (l < D/8)
    // or V row; they go to the cache slot now and into the tile at the last block
    uint4 nkv = make_uint4(0, 0, 0, 0);
    if (cur.slot >= 0 && lane < D / 4) {
      nkv = *reinterpret_cast<const uint4*>(qbuf + 8 * S::kQRow + lane * 8);
      const bool isv = lane >= D / 8;
      const int c = isv ? lane - D / 8 : lane;
      const size_t dst = ((size_t(cur.slot / kBlockSize) * Hkv + g) * kBlockSize +
                          size_t(cur.slot % kBlockSize)) * (D / 8) + c;
      static_cast<uint4*>(const_cast<void*>(isv ? p.v_cache : p.k_cache))[dst] = nkv;
    }
    // kUnitOwn: lane l < D/4 loads 16 bytes of member i's new K row (l < D/8)
    // or V row, used when the member's last block is patched and stored to
    // its slot after the item (its own blocks are at the item's end, so the
    // loads have the shared blocks' time to land)
    uint4 mkv[NT == 2 ? kAbsorbMembers : 1];
#pragma unroll
    for (int i = 0; i < (NT == 2 ? kAbsorbMembers : 1); ++i) {
      mkv[i] = make_uint4(0, 0, 0, 0);
      if (NT == 2 && ((cur.okmask >> i) & 1u) && lane < D / 4) {
        const bool isv = lane >= D / 8;
        const int c = isv ? lane - D / 8 : lane;
        mkv[i] = __ldg(static_cast<const uint4*>(isv ? p.v_new : p.k_new) +
                       (size_t(b + i) * Hkv + g) * (D / 8) + c);
      }
    }
    // qbuf is read: order those reads before the copy that refills it
    dev::fence_proxy_async_smem();
    __syncwarp();
    if (nblk - cur_issued <= kLead) request();
    top_up(kc);

    // per row tile t: O^T accumulators, and the running max / sum of its
    // two query columns (n0, n0 + 1) held by this lane
    float o[NT][KT][4];
    float m0[NT], m1[NT], l0[NT], l1[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) o[t][mt][0] = o[t][mt][1] = o[t][mt][2] = o[t][mt][3] = 0.f;
      m0[t] = m1[t] = -INFINITY;
      l0[t] = l1[t] = 0.f;
    }
    const float sl2 = p.scale_log2;
    // lane 0: how many of the other splits of (b, g) had arrived when this
    // one started its last block (read then, used at the end)
    int seen = -1;

    for (int j = 0; j < nblk; ++j) {
      const int st = cst;
      if (NT == 1 && j == nblk - 1 && nsplit > 1 && lane == 0)
        seen = dev::ld_relaxed_gpu(&p.ws.arrivals[size_t(b) * Hkv + g]);
      if (!mbar_wait_bounded(&my_full[st], cph, tmo, p.status)) {
        drain();
        return;
      }
      const uint32_t kt = dev::smem_u32(ring + size_t(st) * S::kStageBytes);
      const uint32_t vt = kt + S::kTileBytes;
      // the block's member (-1: every row), tokens in context, patch row
      int bmem = -1, bval = ctx - (first + j) * kBlockSize;
      if constexpr (NT == 2) {
        if (cur.flags & kUnitOwn) {
          bmem = __shfl_sync(0xffffffffu, cur.bmem, j);
          bval = __shfl_sync(0xffffffffu, cur.bvalid, j);
          const int bpr = __shfl_sync(0xffffffffu, cur.bpatch, j);
          if (bpr >= 0) {
            // member bmem's new token replaces whatever its slot held
            uint4 v = mkv[0];
#pragma unroll
            for (int i = 1; i < kAbsorbMembers; ++i)
              if (bmem == i) v = mkv[i];
            if (lane < D / 4) {
              const bool isv = lane >= D / 8;
              const int c = isv ? lane - D / 8 : lane;
              const uint32_t addr =
                  (isv ? vt : kt) + (c >> 3) * 2048 + bpr * 128 + (((c & 7) ^ (bpr & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                           "r"(v.y), "r"(v.z), "r"(v.w)
                           : "memory");
            }
            __syncwarp();
          }
        }
      }
      if (cur.patch && j == nblk - 1) {
        // the new token's row replaces whatever the cache held at its slot
        const int r = (ctx - 1) % kBlockSize;
        if (lane < D / 4) {
          const bool isv = lane >= D / 8;
          const int c = isv ? lane - D / 8 : lane;
          const uint32_t addr =
              (isv ? vt : kt) + (c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(nkv.x),
                       "r"(nkv.y), "r"(nkv.z), "r"(nkv.w)
                       : "memory");
        }
        __syncwarp();
      }
      // ---- S^T (16 tokens x 8 rows) = K (16 x D) . Q^T (D x 8), per row tile
      float sa[NT][4], sb[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t)
        sa[t][0] = sa[t][1] = sa[t][2] = sa[t][3] = sb[t][0] = sb[t][1] = sb[t][2] = sb[t][3] = 0.f;
      {
        const int row = lane & 15;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          const int gc = 2 * kk + (lane >> 4);  // 16-byte chunk along head_dim
          const uint32_t addr =
              kt + (gc >> 3) * 2048 + row * 128 + ((((gc & 7) ^ (row & 7))) << 4);
          uint32_t a0, a1, a2, a3;
          dev::ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t == 1 && !two) continue;
            if (kk & 1)
              M::run(sb[t], a0, a1, a2, a3, qb0[t][kk], qb1[t][kk]);
            else
              M::run(sa[t], a0, a1, a2, a3, qb0[t][kk], qb1[t][kk]);
          }
        }
      }
      // ---- mask, scale to base 2, online softmax per query column
      const int valid = bval;  // tokens of the block in context
      const int r0 = lane >> 2;
      const bool v0 = r0 < valid, v1 = r0 + 8 < valid;
      uint32_t pb0[NT], pb1[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t == 1 && !two) {
          pb0[t] = pb1[t] = 0u;
          continue;
        }
        // a member's own block counts for that member's rows only
        const bool c0 = bmem < 0 || mc0[t] == bmem, c1 = bmem < 0 || mc1[t] == bmem;
        const float x0 = v0 && c0 ? (sa[t][0] + sb[t][0]) * sl2 : -INFINITY;
        const float x1 = v0 && c1 ? (sa[t][1] + sb[t][1]) * sl2 : -INFINITY;
        const float x2 = v1 && c0 ? (sa[t][2] + sb[t][2]) * sl2 : -INFINITY;
        const float x3 = v1 && c1 ? (sa[t][3] + sb[t][3]) * sl2 : -INFINITY;
        float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o_));
          bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o_));
        }
        const float mn0 = fmaxf(m0[t], bm0), mn1 = fmaxf(m1[t], bm1);
        const float al0 = dev::fast_exp2(m0[t] - mn0), al1 = dev::fast_exp2(m1[t] - mn1);
        m0[t] = mn0;
        m1[t] = mn1;
        const uint32_t p01 = M::pack(dev::fast_exp2(x0 - mn0), dev::fast_exp2(x1 - mn1));
        const uint32_t p23 = M::pack(dev::fast_exp2(x2 - mn0), dev::fast_exp2(x3 - mn1));
        {
          const float2 f01 = M::unpack(p01), f23 = M::unpack(p23);
          l0[t] = l0[t] * al0 + f01.x + f23.x;
          l1[t] = l1[t] * al1 + f01.y + f23.y;
        }
        // rescale O only when some column's running max grew (x 1 is exact;
        // with two row tiles the multiplies are a good share of the block)
        if (NT == 1 || __any_sync(0xffffffffu, al0 < 1.f || al1 < 1.f)) {
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            o[t][mt][0] *= al0;
            o[t][mt][1] *= al1;
            o[t][mt][2] *= al0;
            o[t][mt][3] *= al1;
          }
        }
        // ---- P^T as the B operand: transpose the two 8x8 halves in registers
        pb0[t] = dev::movmatrix_trans(p01);
        pb1[t] = dev::movmatrix_trans(p23);
      }
      // V^T fragments hold tokens 2(lane%4)+{0,1} (a0, a1) and +8 (a2, a3):
      // zero the ones past the context so their bits never meet P = 0.
      uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
      if (valid < kBlockSize) {
        const int t = 2 * (lane & 3);
        vm_lo = (t < valid ? 0x0000ffffu : 0u) | (t + 1 < valid ? 0xffff0000u : 0u);
        vm_hi = (t + 8 < valid ? 0x0000ffffu : 0u) | (t + 9 < valid ? 0xffff0000u : 0u);
      }
      // ---- O^T (D x 8) += V^T (D x 16 tokens) . P^T (16 tokens x 8), per row tile
      // (a block full of context, all but a sequence's last, takes no masks)
      auto pv = [&](auto masked) {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          const int gc = 2 * mt + ((lane >> 3) & 1);
          const uint32_t addr =
              vt + (gc >> 3) * 2048 + tok * 128 + ((((gc & 7) ^ (tok & 7))) << 4);
          uint32_t a0, a1, a2, a3;
          dev::ldmatrix_x4_trans(addr, a0, a1, a2, a3);
          if constexpr (decltype(masked)::value) {
            a0 &= vm_lo;
            a1 &= vm_lo;
            a2 &= vm_hi;
            a3 &= vm_hi;
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t == 1 && !two) continue;
            M::run(o[t][mt], a0, a1, a2, a3, pb0[t], pb1[t]);
          }
        }
      };
      if (valid < kBlockSize)
        pv(std::true_type{});
      else
        pv(std::false_type{});
      // the stage is read; order those reads before the copy that reuses it
      dev::fence_proxy_async_smem();
      __syncwarp();
      ++kc;
      if (++cst == NS) {
        cst = 0;
        cph ^= 1;
      }
      advance();
      if (cstage == 0 && nblk - cur_issued <= kLead) request();
      top_up(kc);
    }

    // ---- end of the item: this warp holds the whole (m, l, O) of its split
    if constexpr (NT == 1) {
#pragma unroll
      for (int o_ = 4; o_ < 32; o_ <<= 1) {
        l0[0] += __shfl_xor_sync(0xffffffffu, l0[0], o_);
        l1[0] += __shfl_xor_sync(0xffffffffu, l1[0], o_);
      }
      const int n0 = 2 * (lane & 3), n1 = n0 + 1;
      const float inv0 = 1.f / l0[0], inv1 = 1.f / l1[0];
      const size_t head0 = size_t(b) * Hq + size_t(g) * G;
      if (nsplit == 1 && p.cas_o) {
        float* crow = p.cas_o + head0 * D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          const int d0 = 16 * mt + (lane >> 2);
          if (n0 < G) {
            crow[n0 * D + d0] = o[0][mt][0] * inv0;
            crow[n0 * D + d0 + 8] = o[0][mt][2] * inv0;
          }
          if (n1 < G) {
            crow[n1 * D + d0] = o[0][mt][1] * inv1;
            crow[n1 * D + d0 + 8] = o[0][mt][3] * inv1;
          }
        }
        if (lane < 4) {
          if (n0 < G) p.cas_lse[head0 + n0] = m0[0] + log2f(l0[0]);
          if (n1 < G) p.cas_lse[head0 + n1] = m1[0] + log2f(l1[0]);
        }
      } else if (nsplit == 1) {
        T* orow = static_cast<T*>(p.out) + head0 * D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          const int d0 = 16 * mt + (lane >> 2);
          if (n0 < G) {
            orow[n0 * D + d0] = M::from_float(o[0][mt][0] * inv0);
            orow[n0 * D + d0 + 8] = M::from_float(o[0][mt][2] * inv0);
          }
          if (n1 < G) {
            orow[n1 * D + d0] = M::from_float(o[0][mt][1] * inv1);
            orow[n1 * D + d0 + 8] = M::from_float(o[0][mt][3] * inv1);
          }
        }
      } else {
        const size_t part0 = (size_t(b) * p.max_splits + s) * Hq + size_t(g) * G;
        float* prow = p.ws.part_o + part0 * D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          const int d0 = 16 * mt + (lane >> 2);
          if (n0 < G) {
            prow[n0 * D + d0] = o[0][mt][0] * inv0;
            prow[n0 * D + d0 + 8] = o[0][mt][2] * inv0;
          }
          if (n1 < G) {
            prow[n1 * D + d0] = o[0][mt][1] * inv1;
            prow[n1 * D + d0 + 8] = o[0][mt][3] * inv1;
          }
        }
        if (lane < 4) {
          if (n0 < G) p.ws.part_lse[part0 + n0] = m0[0] + log2f(l0[0]);
          if (n1 < G) p.ws.part_lse[part0 + n1] = m1[0] + log2f(l1[0]);
        }
        // Publish this split and count it (release); the warp that completes
        // (b, g) sees every other split's results (acquire) and merges them.
        // If every other split had already arrived when this one began its
        // last block, this one is the last: it acquires their results with a
        // fence and merges without counting itself (nothing else reads the
        // counter in this run), saving the release and the add's round trip.
        const bool alone = __shfl_sync(0xffffffffu, seen, 0) == nsplit - 1;
        if (alone && lane == 0) dev::fence_acq_rel_gpu();
        __syncwarp();
        int last = alone;
        if (!alone) {
          if (lane == 0)
            last = dev::atom_add_acq_rel_gpu(&p.ws.arrivals[size_t(b) * Hkv + g], 1) == nsplit - 1;
          last = __shfl_sync(0xffffffffu, last, 0);
        }
        if (last) {
#ifdef PA_PROFILE_TIMES
          const unsigned long long merge_t0 = dev::global_timer_ns();
#endif
          __syncwarp();
          const size_t row0 = size_t(b) * p.max_splits * Hq + size_t(g) * G;
          MergeArgs ma;
          ma.lse = p.ws.part_lse + row0;
          ma.po = reinterpret_cast<const float4*>(p.ws.part_o + row0 * D);
          ma.out = static_cast<T*>(p.out) + head0 * D;
          ma.cas_o = p.cas_o ? p.cas_o + head0 * D : nullptr;
          ma.cas_lse = p.cas_lse ? p.cas_lse + head0 : nullptr;
          ma.G = G;
          ma.Hq = Hq;
          ma.nsplit = nsplit;
          merge_dispatch<T, D, 24>(ma, lane);
          if (lane == 0) p.ws.arrivals[size_t(b) * Hkv + g] = 0;  // ready for the next run
#ifdef PA_PROFILE_TIMES
          merge_ns = dev::global_timer_ns() - merge_t0;
#endif
        }
      }
    } else {
      // Rows of several members: row r belongs to sequence b + r / G, query
      // head g G + r % G, and each member has its own split count.  A
      // member's only split writes its output; otherwise the split's result
      // goes to the member's split slot for the member's merge.
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
          l0[t] += __shfl_xor_sync(0xffffffffu, l0[t], o_);
          l1[t] += __shfl_xor_sync(0xffffffffu, l1[t], o_);
        }
      }
      const int n0 = 2 * (lane & 3);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t == 1 && !two) continue;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int r = 8 * t + n0 + c;
          if (r >= rows) continue;
          const int bi = b + r / G, head = g * G + r % G;
          const int nsi = r < G ? nsplit : __ldg(&p.ws.nsplits[bi]);
          const float lsum = c ? l1[t] : l0[t];
          const float inv = 1.f / lsum;
          const float lse = (c ? m1[t] : m0[t]) + log2f(lsum);
          const size_t hrow = size_t(bi) * Hq + head;
          if (nsi == 1 && p.cas_o) {
            float* crow = p.cas_o + hrow * D;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
              const int d0 = 16 * mt + (lane >> 2);
              crow[d0] = o[t][mt][c] * inv;
              crow[d0 + 8] = o[t][mt][2 + c] * inv;
            }
            if (lane < 4) p.cas_lse[hrow] = lse;
          } else if (nsi == 1) {
            T* orow = static_cast<T*>(p.out) + hrow * D;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
              const int d0 = 16 * mt + (lane >> 2);
              orow[d0] = M::from_float(o[t][mt][c] * inv);
              orow[d0 + 8] = M::from_float(o[t][mt][2 + c] * inv);
            }
          } else if (team) {
            // the team merges from shared memory: rows kTeamRow floats apart
            float* area = reinterpret_cast<float*>(ring);
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
              const int d0 = 16 * mt + (lane >> 2);
              area[r * kTeamRow + d0] = o[t][mt][c] * inv;
              area[r * kTeamRow + d0 + 8] = o[t][mt][2 + c] * inv;
            }
            if (lane < 4) area[16 * kTeamRow + r] = lse;
          } else if (s >= p.max_splits) {
            dev::flag_status(p.status, kStatusBounds);  // (the plan never makes so many)
          } else {
            const size_t part = (size_t(bi) * p.max_splits + s) * Hq + head;
            float* prow = p.ws.part_o + part * D;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
              const int d0 = 16 * mt + (lane >> 2);
              prow[d0] = o[t][mt][c] * inv;
              prow[d0 + 8] = o[t][mt][2 + c] * inv;
            }
            if (lane < 4) p.ws.part_lse[part] = lse;
          }
        }
      }
      // the members' new tokens go to their slots (kUnitOwn; attended above)
#pragma unroll
      for (int i = 0; i < kAbsorbMembers; ++i) {
        const long long ms = __shfl_sync(0xffffffffu, cur.mslot, i);
        if (((cur.okmask >> i) & 1u) && lane < D / 4) {
          const bool isv = lane >= D / 8;
          const int c = isv ? lane - D / 8 : lane;
          const size_t dst = ((size_t(ms / kBlockSize) * Hkv + g) * kBlockSize +
                              size_t(ms % kBlockSize)) * (D / 8) + c;
          static_cast<uint4*>(const_cast<void*>(isv ? p.v_cache : p.k_cache))[dst] = mkv[i];
        }
      }
      // Count this split in for each of its members with several; the
      // member's last split queues the member's merge, which a warp that
      // has run out of items takes (after the item loop).  (Teams merge
      // after the item loop, from shared memory.)
      __syncwarp();
      if (!team && lane < cur.m) {
        const int bi = b + lane;
        const int nsi = lane == 0 ? nsplit : __ldg(&p.ws.nsplits[bi]);
        if (nsi > 1) {
          const int pair = bi * Hkv + g;
          if (dev::atom_add_acq_rel_gpu(&p.ws.arrivals[pair], 1) == nsi - 1) {
            p.ws.arrivals[pair] = 0;  // ready for the next run
            const int at = atomicAdd(&p.ws.header[kHdrQTail], 1);
            if (at < p.num_seqs * Hkv)
              dev::st_release_gpu(&p.ws.mqueue[at], pair + 1);
            else
              dev::flag_status(p.status, kStatusBounds);
          }
        }
      }
    }
#ifdef PA_PROFILE_TIMES
    ITEM_TRACE(n_items, item_t0, nblk, nsplit, merge_ns, qwait_ns);
    ++n_items;
#endif
    // the next item must be complete before it becomes the current one
    if (cstage == 0) request();
    while (cstage != 4) advance();
  }
  if constexpr (NT == 2) {
    if (team && planned) {
      // Every warp of the team is here (an item of its own done, or none):
      // member j of the team's (chunk, KV head) is merged by the team's
      // warp j from the splits' rows in the team's rings.
      uint64_t* tbar = &team_bars[warp / kTeamWarps];
      if (lane == 0) dev::mbar_arrive(tbar);
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(tbar, 0, tmo, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();  // every lane reads the team's rings after lane 0's acquire
      const int t = (warp / kTeamWarps) * int(gridDim.x) + int(blockIdx.x);
      const int j = warp % kTeamWarps;
      if (ok && t * kTeamWarps < total) {
        const int gg = t % Hkv;
        const int4 u0 = __ldg(&units[(t / Hkv) * kTeamWarps]);
        const int b0 = u0.x, m = (u0.z >> 8) & 0xff;
        if (b0 >= 0 && j < m && b0 + j < p.num_seqs) {
          const int ns = __ldg(&p.ws.nsplits[b0 + j]);
          if (ns > 1 && ns <= kTeamWarps)
            team_merge<T, D>(smem + size_t(warp - j) * NS * S::kStageBytes,
                             size_t(NS) * S::kStageBytes, ns, j * G, G,
                             static_cast<T*>(p.out) + (size_t(b0 + j) * Hq + size_t(gg) * G) * D,
                             lane);
          else if (ns > kTeamWarps && lane == 0)
            dev::flag_status(p.status, kStatusBounds);
        }
      }
    } else if (planned) {
      // The queued merges: every warp out of items takes entries in turn,
      // waits for each to be filled and merges that (sequence, KV head).
      // All items are claimed by then, so each awaited entry is filled by a
      // warp still at work on one (none waits on a warp that waits).
      const int merges = *reinterpret_cast<volatile int*>(&p.ws.header[kHdrMerges]);
      const int cap = p.num_seqs * Hkv;
      for (;;) {
        int at = 0;
        if (lane == 0) at = atomicAdd(&p.ws.header[kHdrQHead], 1);
        at = __shfl_sync(0xffffffffu, at, 0);
        if (at >= merges || at >= cap) break;
        int v = 0;
        if (lane == 0) v = dev::wait_nonzero_bounded(&p.ws.mqueue[at], tmo, p.status);
        v = __shfl_sync(0xffffffffu, v, 0);
        if (v <= 0 || v > cap) {
          if (v > cap && lane == 0) dev::flag_status(p.status, kStatusBounds);
          break;  // (v == 0: the wait ran out and set the status)
        }
        __syncwarp();
        const int bb = (v - 1) / Hkv, gg = (v - 1) % Hkv;
        const int nsi = __ldg(&p.ws.nsplits[bb]);
        if (nsi > 1 && nsi <= p.max_splits) {
          const size_t row0 = size_t(bb) * p.max_splits * Hq + size_t(gg) * G;
          MergeArgs ma;
          ma.lse = p.ws.part_lse + row0;
          ma.po = reinterpret_cast<const float4*>(p.ws.part_o + row0 * D);
          ma.out = static_cast<T*>(p.out) + (size_t(bb) * Hq + size_t(gg) * G) * D;
          ma.cas_o = nullptr;
          ma.cas_lse = nullptr;
          ma.G = G;
          ma.Hq = Hq;
          ma.nsplit = nsi;
          merge_dispatch<T, D, 24>(ma, lane);
        } else if (lane == 0) {
          dev::flag_status(p.status, kStatusBounds);
        }
        if (lane == 0) p.ws.mqueue[at] = 0;  // ready for the next run
      }
      // the last warp done with the queue leaves it ready for the next run
      if (lane == 0 && atomicAdd(&p.ws.header[kHdrQDone], 1) == nwarps - 1) {
        p.ws.header[kHdrQHead] = 0;
        p.ws.header[kHdrQTail] = 0;
        p.ws.header[kHdrQDone] = 0;
      }
    }
  }
  TIME_MARK(1, dev::global_timer_ns());
  TIME_MARK(2, static_cast<unsigned long long>(kc));
}


// --------------------------------------------------------------- fp32 path
template <int D>
__global__ void __launch_bounds__(128) decode_f32_kernel(const Params p) {
  constexpr int E = D / 32;  // consecutive head_dim elements per lane
  const int unit = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (unit >= p.num_seqs * p.num_q_heads) return;
  const int b = unit / p.num_q_heads, h = unit % p.num_q_heads;
  const int g = h / p.group;
  const int cap = p.max_blocks * kBlockSize;
  int ctx = p.context_lens[b];
  if (ctx < 0 || ctx > cap) {
    if (lane == 0) dev::flag_status(p.status, kStatusBounds);
    ctx = ctx < 0 ? 0 : cap;
  }
  const float* qv = static_cast<const float*>(p.q) + (size_t(b) * p.num_q_heads + h) * D + lane * E;
  const float* k_cache = static_cast<const float*>(p.k_cache);
  const float* v_cache = static_cast<const float*>(p.v_cache);
  const int32_t* table = p.block_tables + size_t(b) * p.max_blocks;
  float qr[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qr[e] = qv[e];
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int t = 0; t < ctx; ++t) {
    int phys = table[t / kBlockSize];
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) dev::flag_status(p.status, kStatusBounds);
      phys = 0;
    }
    const size_t row =
        ((size_t(phys) * p.num_kv_heads + g) * kBlockSize + t % kBlockSize) * D + lane * E;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(qr[e], k_cache[row + e], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float sc = dot * p.scale;
    const float mn = fmaxf(m, sc);
    const float a = expf(m - mn), pw = expf(sc - mn);
    l = l * a + pw;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = acc[e] * a + pw * v_cache[row + e];
    m = mn;
  }
  float* out = static_cast<float*>(p.out) + (size_t(b) * p.num_q_heads + h) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = ctx > 0 ? acc[e] / l : 0.f;
}

}  // namespace decode
}  // namespace pa

namespace pa {
namespace decode {

// Last step of a shared-prefix decode: each (sequence, head) merges the
// shared prefix's (o, lse) with its own suffix's by log-sum-exp weights
// (base 2); a side empty of tokens has lse = -inf and weight 0.  Also checks
// that every table starts with the shared prefix (row 0's entries; none with
// prefix_blocks 0).  Grouped mode (seq_blocks non-null): the row's parts are
// those of its own group's prefix (seq_blocks[b] blocks, split as the word
// at split_blocks says); the tables were checked when the step was planned.
template <typename T, int D>
__global__ void __launch_bounds__(256)
    cascade_combine_kernel(const float* __restrict__ po, const float* __restrict__ plse,
                           const int* __restrict__ prefix_parts, const float* __restrict__ so,
                           const float* __restrict__ slse, T* out, int rows,
                           const int32_t* __restrict__ block_tables, int prefix_blocks,
                           int num_seqs, int max_blocks, unsigned* status,
                           const int* __restrict__ seq_blocks, const int* __restrict__ split_blocks,
                           int num_q_heads) {
  dev::grid_dependency_wait();
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = tid; i < (long long)num_seqs * prefix_blocks; i += nthreads) {
    const long long b = i / prefix_blocks, j = i % prefix_blocks;
    if (block_tables[b * max_blocks + j] != block_tables[j]) dev::flag_status(status, kStatusBounds);
  }
  // the prefix phase's parts per row: 1 .. kSharedMaxSplits (part k of row r
  // at po + (k * rows + r) * D, plse[k * rows + r]); 0 in grouped mode for a
  // group with no shared blocks
  int np_all = seq_blocks ? 0 : *prefix_parts;
  if (!seq_blocks && (np_all < 1 || np_all > prefill::kSharedMaxSplits)) {
    if (tid == 0) dev::flag_status(status, kStatusBounds);
    np_all = np_all < 1 ? 1 : prefill::kSharedMaxSplits;
  }
  const int split = seq_blocks ? *split_blocks : 0;
  using M = dev::Mma<T>;
  const int lane = threadIdx.x & 31;
  for (long long r = tid >> 5; r < rows; r += nthreads >> 5) {
    const int np = seq_blocks ? prefill::shared_prefix_parts(seq_blocks[r / num_q_heads], split)
                              : np_all;
    // weights of the prefix parts and of the suffix, by their log-sum-exp
    float lp[prefill::kSharedMaxSplits];
    const float ls = slse[r];
    float m = ls;
#pragma unroll
    for (int k = 0; k < prefill::kSharedMaxSplits; ++k) {
      lp[k] = k < np ? plse[size_t(k) * rows + r] : -INFINITY;
      m = fmaxf(m, lp[k]);
    }
    float wp[prefill::kSharedMaxSplits], sum = 0.f;
#pragma unroll
    for (int k = 0; k < prefill::kSharedMaxSplits; ++k) {
      wp[k] = lp[k] == -INFINITY ? 0.f : dev::fast_exp2(lp[k] - m);
      sum += wp[k];
    }
    const float ws = ls == -INFINITY ? 0.f : dev::fast_exp2(ls - m);
    sum += ws;
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int c = 4 * lane; c < D; c += 128) {
      const float4 b = *reinterpret_cast<const float4*>(so + r * D + c);
      float4 acc = make_float4(ws * b.x, ws * b.y, ws * b.z, ws * b.w);
#pragma unroll
      for (int k = 0; k < prefill::kSharedMaxSplits; ++k) {
        if (k < np) {
          const float4 a = *reinterpret_cast<const float4*>(po + (size_t(k) * rows + r) * D + c);
          acc.x += wp[k] * a.x;
          acc.y += wp[k] * a.y;
          acc.z += wp[k] * a.z;
          acc.w += wp[k] * a.w;
        }
      }
      uint2 pk;
      pk.x = M::pack(acc.x * inv, acc.y * inv);
      pk.y = M::pack(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(out + r * D + c) = pk;
    }
  }
}

// Grouped shared-prefix decode, once per step: CTA b finds sequence b's group
// (the g with group_start[g] <= b < group_start[g + 1]), checks that its table
// starts with the group's prefix (the first member's first group_blocks[g]
// entries), and writes what the suffix decode and the combine read: the
// table past the prefix (-1 padded), the context past it, and the prefix's
// block count.  Bad groups or lengths set the status word (the sequence then
// keeps no prefix).
__global__ void __launch_bounds__(128)
    grouped_suffix_kernel(const int32_t* __restrict__ block_tables,
                          const int32_t* __restrict__ context_lens,
                          const int32_t* __restrict__ group_start,
                          const int32_t* __restrict__ group_blocks, int num_groups, int num_seqs,
                          int max_blocks, int32_t* __restrict__ sfx_tables,
                          int32_t* __restrict__ sfx_ctx, int32_t* __restrict__ seq_blocks,
                          unsigned* status) {
  __shared__ int s_nb, s_first;
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();  // the previous kernel may still read these arrays
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    if (b == 0) {
      bool ok = group_start[0] == 0 && group_start[num_groups] == num_seqs;
      for (int g = 0; g < num_groups && ok; ++g) ok = group_start[g] <= group_start[g + 1];
      if (!ok) dev::flag_status(status, kStatusBounds);
    }
    int lo = 0, hi = num_groups - 1;  // the last g with group_start[g] <= b
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (group_start[mid] <= b) lo = mid;
      else hi = mid - 1;
    }
    const int first = group_start[lo];
    int nb = group_blocks[lo];
    const int ctx = context_lens[b];
    if (first > b || group_start[lo + 1] <= b || first < 0 || nb < 0 || nb > max_blocks ||
        ctx < nb * kBlockSize || ctx > max_blocks * kBlockSize) {
      dev::flag_status(status, kStatusBounds);
      nb = 0;
    }
    s_nb = nb;
    s_first = first < 0 || first >= num_seqs ? b : first;
    sfx_ctx[b] = max(0, min(ctx, max_blocks * kBlockSize) - nb * kBlockSize);
    seq_blocks[b] = nb;
  }
  __syncthreads();
  const int nb = s_nb, first = s_first;
  const int32_t* row = block_tables + size_t(b) * max_blocks;
  for (int j = threadIdx.x; j < max_blocks; j += blockDim.x) {
    if (j < nb && row[j] != block_tables[size_t(first) * max_blocks + j])
      dev::flag_status(status, kStatusBounds);
    sfx_tables[size_t(b) * max_blocks + j] = j + nb < max_blocks ? row[j + nb] : -1;
  }
}

}  // namespace decode
}  // namespace pa

// ====================================================================== host
namespace pa {
namespace decode {
namespace {

constexpr int kMaxDevices = 64;

struct KernelConfig {
  int stages = 0;
  int ctas_per_sm = 0;
  size_t smem = 0;
};

// Tuning knobs read once per process: math warps per CTA (4 or 8), CTAs per
// SM, and a cap on the ring stages per math warp.  Defaults are the measured
// best.
struct Tuning {
  int split_blocks = 0;  // 0: kSplitBlocks (measured best for both MHA and GQA batches)
  int warps = kConsumerWarps;
  int ctas_per_sm = 1;
  int max_stages = kWarpStages;
  int tail_waves = kTailWaves;
  int piece_blocks = kPieceBlocks;
};
Tuning read_tuning_env() {
  Tuning t;
  if (const char* v = std::getenv("PA_DECODE_WARPS")) t.warps = std::atoi(v) == 4 ? 4 : 8;
  if (const char* v = std::getenv("PA_DECODE_SPLIT_BLOCKS"))
    t.split_blocks = std::max(kMinSplitBlocks, std::min(kSplitBlocks, std::atoi(v)));
  if (const char* v = std::getenv("PA_DECODE_CTAS_PER_SM")) t.ctas_per_sm = std::max(1, std::min(4, std::atoi(v)));
  if (const char* v = std::getenv("PA_DECODE_MAX_STAGES")) t.max_stages = std::max(1, std::min(kWarpStages, std::atoi(v)));
  if (const char* v = std::getenv("PA_DECODE_TAIL_WAVES")) t.tail_waves = std::max(0, std::min(16, std::atoi(v)));
  if (const char* v = std::getenv("PA_DECODE_PIECE_BLOCKS"))
    t.piece_blocks = std::max(1, std::min(16, std::atoi(v)));
  return t;
}
// Read once per process.
const Tuning& tuning() {
  static const Tuning t = read_tuning_env();
  return t;
}

struct DeviceState {
  std::once_flag once;
  int error = 0;  // PA_OK or the status the set-up failed with
  int sms = 0;
  Tuning tuning;
  KernelConfig cfg[2][2];   // [bf16?][head_dim 128?]
  KernelConfig cfg2[2][2];  // the same for two query-row tiles (grouped decode, 8 warps)
};
DeviceState g_dev[kMaxDevices];


template <typename T, int D, int W, int NT = 1>
cudaError_t configure_kernel(KernelConfig* cfg, const Tuning& t, size_t optin, size_t per_sm) {
  // shared memory per CTA when `ctas_per_sm` CTAs share an SM (1 KiB reserved each)
  size_t budget = per_sm / t.ctas_per_sm - 1024;
  if (budget > optin) budget = optin;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, W, NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(budget));
  if (e != cudaSuccess) return e;
  int stages = Smem<D, W, NT>::stages_for(budget);  // per math warp
  if (stages > t.max_stages) stages = t.max_stages;
  cfg->stages = stages;
  cfg->smem = Smem<D, W, NT>::bytes(stages);
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cfg->ctas_per_sm,
                                                    decode_kernel<T, D, W, NT>, W * 32, cfg->smem);
  if (cfg->ctas_per_sm > t.ctas_per_sm) cfg->ctas_per_sm = t.ctas_per_sm;
  return e;
}

template <int W>
cudaError_t configure_all(DeviceState& st, size_t optin, size_t per_sm) {
  cudaError_t e = configure_kernel<__nv_bfloat16, 128, W>(&st.cfg[1][1], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__nv_bfloat16, 64, W>(&st.cfg[1][0], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__half, 128, W>(&st.cfg[0][1], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__half, 64, W>(&st.cfg[0][0], st.tuning, optin, per_sm);
  // the grouped decode always runs 8 math warps per CTA
  if (e == cudaSuccess)
    e = configure_kernel<__nv_bfloat16, 128, 8, 2>(&st.cfg2[1][1], st.tuning, optin, per_sm);
  if (e == cudaSuccess)
    e = configure_kernel<__nv_bfloat16, 64, 8, 2>(&st.cfg2[1][0], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__half, 128, 8, 2>(&st.cfg2[0][1], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__half, 64, 8, 2>(&st.cfg2[0][0], st.tuning, optin, per_sm);
  return e;
}

int device_setup(int device) {
  DeviceState& st = g_dev[device];
  std::call_once(st.once, [&] {
    int optin = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) !=
            cudaSuccess) {
      st.error = PA_ERR_CUDA;
      return;
    }
    st.tuning = tuning();
    cudaError_t e = st.tuning.warps == 4 ? configure_all<4>(st, optin, per_sm)
                                         : configure_all<8>(st, optin, per_sm);
    st.error = e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    for (int a = 0; a < 2 && st.error == PA_OK; ++a)
      for (int d = 0; d < 2; ++d)
        if (st.cfg[a][d].stages < 1 || st.cfg[a][d].ctas_per_sm < 1 ||
            st.cfg2[a][d].stages < 1 || st.cfg2[a][d].ctas_per_sm < 1)
          st.error = PA_ERR_UNSUPPORTED;
  });
  if (st.error != PA_OK) return fail(st.error, "decode: per-device set-up failed on device %d", device);
  return PA_OK;
}

template <typename T, int D, int W, int NT = 1>
int launch_tc(Params prm, const KernelConfig& kc, int sms, cudaStream_t stream) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  alignas(64) CUtensorMap mk, mv;
  int rc = cache_tensor_map(&mk, prm.k_cache, kBf16, prm.num_blocks, prm.num_kv_heads, D);
  if (rc == PA_OK) rc = cache_tensor_map(&mv, prm.v_cache, kBf16, prm.num_blocks, prm.num_kv_heads, D);
  if (rc != PA_OK) return rc;
  prm.stages = kc.stages;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms * kc.ctas_per_sm);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = kc.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<T, D, W, NT>, mk, mv, prm);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "decode: launch failed: %s", cudaGetErrorString(e));
  return PA_OK;
}

// Host-side checks shared by every decode entry point.
int check_decode_shapes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_blocks_per_seq, int dtype, const char* who) {
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "%s: unknown dtype %d", who, dtype);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d (64 or 128)", who, head_dim);
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: sizes must be positive", who);
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "%s: num_q_heads %% num_kv_heads != 0", who);
  if (dtype != PA_F32 && num_q_heads / num_kv_heads > kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "%s: %d query heads per KV head (max %d)", who,
                num_q_heads / num_kv_heads, kMaxGroup);
  if (double(max_blocks_per_seq) * kBlockSize >= 2147483647.0)
    return fail(PA_ERR_INVALID_ARG, "%s: max_blocks_per_seq too large", who);
  if (layout_too_large(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq))
    return fail(PA_ERR_INVALID_ARG, "%s: these shapes need an impossibly large workspace", who);
  return PA_OK;
}

int check_workspace(void* workspace, size_t workspace_bytes, const Layout& lay, const char* who) {
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "%s: workspace is NULL", who);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (workspace_bytes < lay.total)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                lay.total);
  return PA_OK;
}

Params make_params(const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                   int head_dim, int max_blocks_per_seq, void* workspace, const Layout& lay,
                   unsigned* status) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Params prm = {};
  prm.context_lens = context_lens;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = num_q_heads / num_kv_heads;
  prm.head_dim = head_dim;
  prm.max_blocks = max_blocks_per_seq;
  prm.max_splits = lay.max_splits;
  prm.split_blocks = tuning().split_blocks ? tuning().split_blocks : kSplitBlocks;
  prm.signature = plan_signature(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                 prm.split_blocks);
  prm.ws.header = reinterpret_cast<int*>(ws + lay.header);
  prm.ws.units = reinterpret_cast<int*>(ws + lay.units);
  prm.ws.arrivals = reinterpret_cast<int*>(ws + lay.arrivals);
  prm.ws.nsplits = reinterpret_cast<int*>(ws + lay.nsplits);
  prm.ws.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  prm.ws.part_o = reinterpret_cast<float*>(ws + lay.part_o);
  prm.status = status;
  prm.timeout_ns = 1000000000ull;  // 1 s per wait
  return prm;
}

// Suffix mode of a shared-prefix decode (all zero / null: a plain decode).
struct SuffixArgs {
  int prefix_blocks = 0;
  float* cas_o = nullptr;
  float* cas_lse = nullptr;
};

void apply_suffix(Params& prm, const SuffixArgs& sfx) {
  prm.table_offset = sfx.prefix_blocks;
  prm.ctx_offset = sfx.prefix_blocks * kBlockSize;
  prm.cas_o = sfx.cas_o;
  prm.cas_lse = sfx.cas_lse;
  prm.signature = plan_signature(prm.num_seqs, prm.num_q_heads, prm.num_kv_heads, prm.head_dim,
                                 prm.max_blocks, prm.split_blocks, prm.table_offset);
}

int plan_impl(const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
              int head_dim, int max_blocks_per_seq, void* workspace, size_t workspace_bytes,
              cudaStream_t stream, const char* who, const SuffixArgs& sfx = SuffixArgs()) {
  const Layout lay =
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  int rc = check_workspace(workspace, workspace_bytes, lay, who);
  if (rc != PA_OK) return rc;
  if (!context_lens) return fail(PA_ERR_INVALID_ARG, "%s: context_lens is NULL", who);
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "%s: no current CUDA device", who);
  rc = device_setup(device);
  if (rc != PA_OK) return rc;
  Params prm = make_params(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                           max_blocks_per_seq, workspace, lay, status);
  apply_suffix(prm, sfx);
  // the tail is sized for the math warps the attention kernel will launch
  const DeviceState& st = g_dev[device];
  const int nwarps = st.sms * st.cfg[1][head_dim == 128].ctas_per_sm * st.tuning.warps;
  prm.piece_blocks = st.tuning.piece_blocks;
  prm.tail_blocks = st.tuning.tail_waves * nwarps * prm.piece_blocks;
  static std::once_flag carveout_once;
  std::call_once(carveout_once, [] {
    // keep the SM's shared-memory split the attention kernel wants, so no
    // reconfiguration happens between the plan and the attention kernel
    cudaFuncSetAttribute(plan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, plan_kernel, prm);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: plan launch failed: %s", who, cudaGetErrorString(e));
  return PA_OK;
}

// Host-side checks of the attention launch's own arguments.  Every one-shot
// entry point runs them before its plan, so a call that is rejected leaves
// the workspace untouched.
int check_run_args(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens, const void* out,
                   int num_kv_heads, int num_blocks, const char* who) {
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "%s: num_blocks must be positive", who);
  if (double(num_blocks) * num_kv_heads * kBlockSize >= 2147483647.0)
    return fail(PA_ERR_INVALID_ARG, "%s: cache has too many rows", who);
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out))
    return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", who);
  return PA_OK;
}

// The new tokens a fused call appends (all null: plain attention).
struct AppendArgs {
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* slot_mapping = nullptr;
};

// Checks the new tokens' rows and slots of a fused append call.
int append_args(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                AppendArgs& app, const char* who) {
  if (!k_new || !v_new || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "%s: k_new, v_new and slot_mapping are required", who);
  if ((reinterpret_cast<uintptr_t>(k_new) & 15) || (reinterpret_cast<uintptr_t>(v_new) & 15))
    return fail(PA_ERR_INVALID_ARG, "%s: k_new and v_new must be 16-byte aligned", who);
  app.k_new = k_new;
  app.v_new = v_new;
  app.slot_mapping = slot_mapping;
  return PA_OK;
}

int run_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
             const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
             int head_dim, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
             void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream,
             const char* who, const AppendArgs& app = AppendArgs(),
             const SuffixArgs& sfx = SuffixArgs()) {
  int rc = check_run_args(q, k_cache, v_cache, block_tables, context_lens, out, num_kv_heads,
                          num_blocks, who);
  if (rc != PA_OK) return rc;
  const Layout lay =
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  rc = check_workspace(workspace, workspace_bytes, lay, who);
  if (rc != PA_OK) return rc;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "%s: no current CUDA device", who);
  rc = device_setup(device);
  if (rc != PA_OK) return rc;
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;

  Params prm = make_params(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                           max_blocks_per_seq, workspace, lay, status);
  prm.q = q;
  prm.k_cache = k_cache;
  prm.v_cache = v_cache;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.num_blocks = num_blocks;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  apply_suffix(prm, sfx);

  if (app.slot_mapping && dtype == PA_F32) {
    // the fp32 path is not fused: append first, then attend
    rc = pa_kv_append(app.k_new, app.v_new, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                      app.slot_mapping, num_seqs, num_kv_heads, head_dim, num_blocks, dtype,
                      stream);
    if (rc != PA_OK) return rc;
  } else if (app.slot_mapping) {
    prm.k_new = app.k_new;
    prm.v_new = app.v_new;
    prm.slot_mapping = app.slot_mapping;
  }
  if (dtype == PA_F32) {
    const int blocks = (num_seqs * num_q_heads + 3) / 4;
    if (head_dim == 64)
      decode_f32_kernel<64><<<blocks, 128, 0, stream>>>(prm);
    else
      decode_f32_kernel<128><<<blocks, 128, 0, stream>>>(prm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
      return fail(PA_ERR_CUDA, "%s (fp32): launch failed: %s", who, cudaGetErrorString(e));
    return PA_OK;
  }
  const DeviceState& st = g_dev[device];
  const KernelConfig& kc = st.cfg[dtype == PA_BF16][head_dim == 128];
  if (st.tuning.warps == 4) {
    if (dtype == PA_BF16)
      return head_dim == 128 ? launch_tc<__nv_bfloat16, 128, 4>(prm, kc, st.sms, stream)
                             : launch_tc<__nv_bfloat16, 64, 4>(prm, kc, st.sms, stream);
    return head_dim == 128 ? launch_tc<__half, 128, 4>(prm, kc, st.sms, stream)
                           : launch_tc<__half, 64, 4>(prm, kc, st.sms, stream);
  }
  if (dtype == PA_BF16)
    return head_dim == 128 ? launch_tc<__nv_bfloat16, 128, 8>(prm, kc, st.sms, stream)
                           : launch_tc<__nv_bfloat16, 64, 8>(prm, kc, st.sms, stream);
  return head_dim == 128 ? launch_tc<__half, 128, 8>(prm, kc, st.sms, stream)
                         : launch_tc<__half, 64, 8>(prm, kc, st.sms, stream);
}

}  // namespace
}  // namespace decode
}  // namespace pa

using namespace pa;
using namespace pa::decode;

extern "C" {

#ifdef PA_PROFILE_TIMES
PA_API int pa_profile_item_trace(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, g_item_trace, size_t(n) * sizeof(unsigned long long)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}
PA_API int pa_profile_times(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, g_times, size_t(n) * sizeof(unsigned long long)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}
#endif

PA_API int pa_paged_attention_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                                    int head_dim, int max_blocks_per_seq,
                                                    size_t* bytes) {
  if (!bytes) return fail(PA_ERR_INVALID_ARG, "workspace_size: bytes is NULL");
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "workspace_size: sizes must be positive");
  if (layout_too_large(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq))
    return fail(PA_ERR_INVALID_ARG, "workspace_size: these shapes need an impossibly large workspace");
  *bytes = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total;
  return PA_OK;
}

PA_API int pa_paged_attention_decode_plan(const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_plan");
  const char* who = "paged_attention_decode_plan";
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               PA_BF16, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  return plan_impl(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                   workspace, workspace_bytes, static_cast<cudaStream_t>(stream), who);
}

PA_API int pa_paged_attention_decode_run(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int max_blocks_per_seq, int num_blocks,
                                         float scale, int dtype, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_run");
  const char* who = "paged_attention_decode_run";
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  return run_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                  workspace, workspace_bytes, static_cast<cudaStream_t>(stream), who);
}

PA_API int pa_paged_attention_decode_append_run(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
    int num_blocks, float scale, int dtype, void* out, void* workspace, size_t workspace_bytes,
    void* stream) {
  PA_TRACE("pa_paged_attention_decode_append_run");
  const char* who = "paged_attention_decode_append_run";
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  AppendArgs app;
  rc = append_args(k_new, v_new, slot_mapping, app, who);
  if (rc != PA_OK) return rc;
  return run_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                  workspace, workspace_bytes, static_cast<cudaStream_t>(stream), who, app);
}

}  // extern "C"

namespace {
// Workspace of a shared-prefix decode: the suffix decode's, the prefix
// phase's, then fp32 (o, lse) of both phases.
struct SharedLayout {
  size_t decode, prefix, po, plse, so, slse, total;
};
SharedLayout shared_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int max_blocks_per_seq) {
  SharedLayout l;
  const size_t rows = size_t(num_seqs) * num_q_heads;
  l.decode = 0;
  l.prefix = align256(
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total);
  l.po = align256(l.prefix + prefill::shared_prefix_workspace_bytes(num_seqs, num_q_heads,
                                                                    num_kv_heads, head_dim));
  // the prefix phase may leave up to kSharedMaxSplits parts per row
  l.plse = align256(l.po + size_t(prefill::kSharedMaxSplits) * rows * head_dim * 4);
  l.so = align256(l.plse + size_t(prefill::kSharedMaxSplits) * rows * 4);
  l.slse = align256(l.so + rows * head_dim * 4);
  l.total = align256(l.slse + rows * 4);
  return l;
}

// The grouped cascade adds, per sequence, the table past its group's prefix,
// the context past it and the prefix's block count (written once per step).
struct GroupedLayout {
  SharedLayout sh;
  size_t sfx_tables, sfx_ctx, seq_blocks, total;
};
// Workspace of the one-launch cascade (a grouped decode): the decode
// workspace with one more split per sequence (a sequence's shared splits and
// own splits can round up once each), then each group's checked shared
// blocks, each sequence's shared blocks and its clamped context.
struct FusedLayout {
  Layout dec;
  size_t gp, seq_prefix, seq_ctx, seq_group, seq_chunk, chunk_plan, mqueue, total;
};
FusedLayout fused_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int max_blocks_per_seq) {
  FusedLayout l;
  l.dec = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                           max_blocks_per_seq + kMinSplitBlocks);
  l.gp = l.dec.total;
  l.seq_prefix = align256(l.gp + size_t(num_seqs) * 4 + 4);
  l.seq_ctx = align256(l.seq_prefix + size_t(num_seqs) * 4);
  l.seq_group = align256(l.seq_ctx + size_t(num_seqs) * 4);
  l.seq_chunk = align256(l.seq_group + size_t(num_seqs) * 4);
  l.chunk_plan = align256(l.seq_chunk + size_t(num_seqs) * 8);
  l.mqueue = align256(l.chunk_plan + size_t(num_seqs) * 16);
  l.total = align256(l.mqueue + size_t(num_seqs) * num_kv_heads * 4);
  return l;
}

GroupedLayout grouped_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int max_blocks_per_seq) {
  GroupedLayout l;
  l.sh = shared_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  l.sfx_tables = l.sh.total;
  l.sfx_ctx = align256(l.sfx_tables + size_t(num_seqs) * max_blocks_per_seq * 4);
  l.seq_blocks = align256(l.sfx_ctx + size_t(num_seqs) * 4);
  l.total = align256(l.seq_blocks + size_t(num_seqs) * 4);
  return l;
}
}  // namespace

extern "C" {

PA_API int pa_paged_attention_decode_shared_prefix_workspace_size(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
    size_t* bytes) {
  if (!bytes) return fail(PA_ERR_INVALID_ARG, "shared_prefix_workspace_size: bytes is NULL");
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "shared_prefix_workspace_size: bad sizes");
  if (layout_too_large(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq))
    return fail(PA_ERR_INVALID_ARG,
                "shared_prefix_workspace_size: these shapes need an impossibly large workspace");
  *bytes = std::max(
      shared_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total,
      fused_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total);
  return PA_OK;
}

}  // extern "C"

namespace {

enum class SharedMode { kPlanAndRun, kPlanOnly, kRunOnly };

// Which cascade implementation an entry point uses: the three phases (the
// prefix phase on the chunked-prefill kernels, the suffix decode, the
// combine) or the grouped decode (one attention launch over shared and own
// units, which also merges each sequence's splits).  Measured on GB300
// (8B-shaped GQA): 128 forked branches in groups of 4 sharing 64 blocks took
// 50 us per layer grouped against 52 in phases; 100 requests on one 64-block prefix take 76
// in phases against 91 grouped (the phases read the prefix once for all 400
// query rows; the grouped decode once per 16).  So the grouped entry points
// use the grouped decode and the single-prefix ones the phases;
// PA_CASCADE=phases or =grouped makes every entry point use one of them.
// Read once per process.
enum class CascadeImpl { kDefault, kPhases, kGrouped };
CascadeImpl cascade_impl() {
  static const CascadeImpl impl = [] {
    const char* v = std::getenv("PA_CASCADE");
    if (v && std::strcmp(v, "phases") == 0) return CascadeImpl::kPhases;
    if (v && std::strcmp(v, "grouped") == 0) return CascadeImpl::kGrouped;
    return CascadeImpl::kDefault;
  }();
  return impl;
}

// The one-launch cascade.  group_start == null: one group of every sequence
// sharing `single_blocks` leading blocks.  kPlanOnly reads the lengths, the
// tables and the group arrays (q, the caches and out may be NULL); kRunOnly
// reads the lengths the plan copied into the workspace.
int fused_cascade_impl(SharedMode mode, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                       int single_blocks, int num_seqs, int num_q_heads, int num_kv_heads,
                       int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
                       int dtype, void* out, void* workspace, size_t workspace_bytes,
                       cudaStream_t s, const char* who, const AppendArgs& app) {
  const FusedLayout fl =
      fused_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
      workspace_bytes < fl.total)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace NULL, unaligned or < %zu bytes", who, fl.total);
  const bool plans = mode != SharedMode::kRunOnly, runs = mode != SharedMode::kPlanOnly;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* seq_ctx = reinterpret_cast<int32_t*>(ws + fl.seq_ctx);
  int rc = PA_OK;
  // the grouped plan checks the members' tables; one shared prefix is
  // checked by the run (its plan gets no tables)
  if (plans && (!context_lens || (group_start && !block_tables)))
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (runs) {
    rc = check_run_args(q, k_cache, v_cache, block_tables, seq_ctx, out, num_kv_heads, num_blocks,
                        who);
    if (rc != PA_OK) return rc;
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "%s: no current CUDA device", who);
  rc = device_setup(device);
  if (rc != PA_OK) return rc;
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  const DeviceState& st = g_dev[device];
  const int signature = plan_signature(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                       max_blocks_per_seq,
                                       st.tuning.split_blocks ? st.tuning.split_blocks
                                                              : kSplitBlocks,
                                       0, 1);
  const KernelConfig& kc2 = st.cfg2[dtype == PA_BF16][head_dim == 128];
  if (plans) {
    Params prm = make_params(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                             max_blocks_per_seq, workspace, fl.dec, status);
    prm.block_tables = group_start ? block_tables : nullptr;
    prm.signature = signature;
    prm.ws.mqueue = reinterpret_cast<int*>(ws + fl.mqueue);
    const int nwarps = st.sms * kc2.ctas_per_sm * 8;
    prm.piece_blocks = st.tuning.piece_blocks;
    prm.tail_blocks = st.tuning.tail_waves * nwarps * prm.piece_blocks;
    GroupArgs ga;
    ga.group_start = group_start;
    ga.group_blocks = group_blocks;
    ga.num_groups = group_start ? num_groups : 1;
    ga.single_blocks = single_blocks;
    ga.chunk = 16 / (num_q_heads / num_kv_heads);
    ga.nwarps = nwarps;
    ga.teams = kc2.stages >= 2;  // a split's results fill most of two stages
    ga.small = num_seqs <= kGroupedPlanSmallSeqs && ga.num_groups <= kGroupedPlanSmallSeqs;
    ga.gp = reinterpret_cast<int32_t*>(ws + fl.gp);
    ga.seq_prefix = reinterpret_cast<int32_t*>(ws + fl.seq_prefix);
    ga.seq_ctx = seq_ctx;
    ga.seq_group = reinterpret_cast<int32_t*>(ws + fl.seq_group);
    ga.seq_chunk = reinterpret_cast<int2*>(ws + fl.seq_chunk);
    ga.chunk_plan = reinterpret_cast<int4*>(ws + fl.chunk_plan);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kGroupedPlanThreads);
    cfg.dynamicSmemBytes = ga.small ? grouped_plan_smem(num_seqs, ga.num_groups) : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_plan_kernel, prm, ga);
    if (e != cudaSuccess)
      return fail(PA_ERR_CUDA, "%s: plan launch failed: %s", who, cudaGetErrorString(e));
  }
  if (!runs) return PA_OK;
  Params prm = make_params(seq_ctx, num_seqs, num_q_heads, num_kv_heads, head_dim,
                           max_blocks_per_seq, workspace, fl.dec, status);
  prm.seq_prefix = reinterpret_cast<const int32_t*>(ws + fl.seq_prefix);
  prm.ws.mqueue = reinterpret_cast<int*>(ws + fl.mqueue);
  prm.verify_prefix = group_start == nullptr;
  prm.signature = signature;
  prm.q = q;
  prm.k_cache = k_cache;
  prm.v_cache = v_cache;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.num_blocks = num_blocks;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  if (app.slot_mapping) {
    prm.k_new = app.k_new;
    prm.v_new = app.v_new;
    prm.slot_mapping = app.slot_mapping;
  }
  if (dtype == PA_BF16)
    rc = head_dim == 128 ? launch_tc<__nv_bfloat16, 128, 8, 2>(prm, kc2, st.sms, s)
                         : launch_tc<__nv_bfloat16, 64, 8, 2>(prm, kc2, st.sms, s);
  else
    rc = head_dim == 128 ? launch_tc<__half, 128, 8, 2>(prm, kc2, st.sms, s)
                         : launch_tc<__half, 64, 8, 2>(prm, kc2, st.sms, s);
  if (rc != PA_OK) return rc;
  return PA_OK;
}

// The cascade decode: the prefix phase, each sequence's own blocks, the
// combine.  kPlanOnly launches the two plans (they read only the lengths and
// sizes; q, the caches, the tables and out may be NULL), kRunOnly the three
// compute launches over a planned workspace.
int shared_prefix_impl(SharedMode mode, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, int prefix_blocks,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* out,
                       void* workspace, size_t workspace_bytes, void* stream, const char* who,
                       const AppendArgs& app = AppendArgs()) {
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq)
    return fail(PA_ERR_INVALID_ARG, "%s: prefix_blocks outside 0..max_blocks_per_seq", who);
  const SharedLayout sl =
      shared_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
      workspace_bytes < sl.total)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace NULL, unaligned or < %zu bytes", who, sl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool plans = mode != SharedMode::kRunOnly, runs = mode != SharedMode::kPlanOnly;
  if (!context_lens) return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (runs) {
    rc = check_run_args(q, k_cache, v_cache, block_tables, context_lens, out, num_kv_heads,
                        num_blocks, who);
    if (rc != PA_OK) return rc;
  }
  if (prefix_blocks == 0 || dtype == PA_F32) {
    // nothing shared to exploit (or the fp32 path): a plain decode is exact
    if (plans && dtype != PA_F32) {
      rc = plan_impl(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     max_blocks_per_seq, workspace, workspace_bytes, s, who);
      if (rc != PA_OK) return rc;
    }
    return runs ? run_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                           num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype,
                           out, workspace, workspace_bytes, s, who, app)
                : PA_OK;
  }
  if (runs && (!q || !k_cache || !v_cache || !block_tables || !out))
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (cascade_impl() == CascadeImpl::kGrouped)
    return fused_cascade_impl(mode, q, k_cache, v_cache, block_tables, context_lens, nullptr,
                              nullptr, 1, prefix_blocks, num_seqs, num_q_heads, num_kv_heads,
                              head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                              workspace, workspace_bytes, s, who, app);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* po = reinterpret_cast<float*>(ws + sl.po);
  float* plse = reinterpret_cast<float*>(ws + sl.plse);
  float* so = reinterpret_cast<float*>(ws + sl.so);
  float* slse = reinterpret_cast<float*>(ws + sl.slse);
  SuffixArgs sfx;
  sfx.prefix_blocks = prefix_blocks;
  sfx.cas_o = so;
  sfx.cas_lse = slse;
  if (plans) {
    rc = prefill::shared_prefix_plan(prefix_blocks * kBlockSize, num_seqs, num_q_heads,
                                     num_kv_heads, head_dim, max_blocks_per_seq, scale, dtype,
                                     ws + sl.prefix, sl.po - sl.prefix, s);
    if (rc != PA_OK) return rc;
    rc = plan_impl(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                   workspace, sl.prefix, s, who, sfx);
    if (rc != PA_OK) return rc;
  }
  if (!runs) return PA_OK;
  // 1. the shared prefix, read once for all queries
  rc = prefill::shared_prefix_run(q, k_cache, v_cache, block_tables, prefix_blocks * kBlockSize,
                                  num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  max_blocks_per_seq, num_blocks, scale, dtype, po, plse,
                                  ws + sl.prefix, sl.po - sl.prefix, s);
  if (rc != PA_OK) return rc;
  // 2. every sequence's own blocks (the new tokens, if any, are stored and
  // attended here: they always lie past the shared prefix)
  rc = run_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                workspace, sl.prefix, s, who, app, sfx);
  if (rc != PA_OK) return rc;
  // 3. merge
  const int* parts = prefill::shared_prefix_split_count(ws + sl.prefix);
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  const int rows = num_seqs * num_q_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (dtype == PA_BF16)
    e = head_dim == 128
            ? cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__nv_bfloat16, 128>, po, plse, parts, so,
                                 slse, static_cast<__nv_bfloat16*>(out), rows, block_tables,
                                 prefix_blocks, num_seqs, max_blocks_per_seq, status,
                                 nullptr, nullptr, num_q_heads)
            : cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__nv_bfloat16, 64>, po, plse, parts, so,
                                 slse, static_cast<__nv_bfloat16*>(out), rows, block_tables,
                                 prefix_blocks, num_seqs, max_blocks_per_seq, status,
                                 nullptr, nullptr, num_q_heads);
  else
    e = head_dim == 128
            ? cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__half, 128>, po, plse, parts, so, slse,
                                 static_cast<__half*>(out), rows, block_tables, prefix_blocks,
                                 num_seqs, max_blocks_per_seq, status, nullptr, nullptr,
                                 num_q_heads)
            : cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__half, 64>, po, plse, parts, so, slse,
                                 static_cast<__half*>(out), rows, block_tables, prefix_blocks,
                                 num_seqs, max_blocks_per_seq, status, nullptr, nullptr,
                                 num_q_heads);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: merge launch failed: %s", who, cudaGetErrorString(e));
  return PA_OK;
}

// The grouped cascade: plan (once per step) = the suffix tables and lengths,
// the prefix phase's plan over the groups, the suffix decode's plan; run (per
// layer) = the prefix phase, the suffix decode, the combine.
int grouped_prefix_impl(SharedMode mode, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens,
                        const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* out,
                        void* workspace, size_t workspace_bytes, void* stream, const char* who,
                        const AppendArgs& app = AppendArgs()) {
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (dtype == PA_F32)
    return fail(PA_ERR_UNSUPPORTED, "%s: 16-bit dtypes only (fp32 decodes exactly without it)", who);
  if (num_groups < 1 || num_groups > num_seqs)
    return fail(PA_ERR_INVALID_ARG, "%s: num_groups outside 1..num_seqs", who);
  const GroupedLayout gl =
      grouped_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  const SharedLayout& sl = gl.sh;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
      workspace_bytes < gl.total)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace NULL, unaligned or < %zu bytes", who, gl.total);
  if (!group_start || !group_blocks) return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool plans = mode != SharedMode::kRunOnly, runs = mode != SharedMode::kPlanOnly;
  if (plans && (!context_lens || !block_tables))
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (cascade_impl() != CascadeImpl::kPhases)
    return fused_cascade_impl(mode, q, k_cache, v_cache, block_tables, context_lens, group_start,
                              group_blocks, num_groups, 0, num_seqs, num_q_heads, num_kv_heads,
                              head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                              workspace, workspace_bytes, s, who, app);
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* po = reinterpret_cast<float*>(ws + sl.po);
  float* plse = reinterpret_cast<float*>(ws + sl.plse);
  float* so = reinterpret_cast<float*>(ws + sl.so);
  float* slse = reinterpret_cast<float*>(ws + sl.slse);
  int32_t* sfx_tables = reinterpret_cast<int32_t*>(ws + gl.sfx_tables);
  int32_t* sfx_ctx = reinterpret_cast<int32_t*>(ws + gl.sfx_ctx);
  int32_t* seq_blocks = reinterpret_cast<int32_t*>(ws + gl.seq_blocks);
  if (runs) {
    // the suffix decode reads the suffix lengths the plan writes (a run-only
    // caller passes no context_lens)
    rc = check_run_args(q, k_cache, v_cache, block_tables, sfx_ctx, out, num_kv_heads, num_blocks,
                        who);
    if (rc != PA_OK) return rc;
  }
  SuffixArgs sfx;  // no offsets: the suffix decode reads the suffix tables
  sfx.cas_o = so;
  sfx.cas_lse = slse;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (plans) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_seqs);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_suffix_kernel, block_tables, context_lens,
                                       group_start, group_blocks, num_groups, num_seqs,
                                       max_blocks_per_seq, sfx_tables, sfx_ctx, seq_blocks, status);
    if (e != cudaSuccess)
      return fail(PA_ERR_CUDA, "%s: suffix-table launch failed: %s", who, cudaGetErrorString(e));
    rc = prefill::grouped_prefix_plan(group_start, group_blocks, num_groups, num_seqs, num_q_heads,
                                      num_kv_heads, head_dim, max_blocks_per_seq, scale, dtype,
                                      ws + sl.prefix, sl.po - sl.prefix, s);
    if (rc != PA_OK) return rc;
    rc = plan_impl(sfx_ctx, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                   workspace, sl.prefix, s, who, sfx);
    if (rc != PA_OK) return rc;
  }
  if (!runs) return PA_OK;
  // 1. every group's prefix, read once for the group's queries
  rc = prefill::grouped_prefix_run(q, k_cache, v_cache, block_tables, group_start, group_blocks,
                                   num_groups, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                   max_blocks_per_seq, num_blocks, scale, dtype, po, plse,
                                   ws + sl.prefix, sl.po - sl.prefix, s);
  if (rc != PA_OK) return rc;
  // 2. every sequence's own blocks (and its new token, if any)
  rc = run_impl(q, k_cache, v_cache, sfx_tables, sfx_ctx, num_seqs, num_q_heads, num_kv_heads,
                head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out, workspace, sl.prefix,
                s, who, app, sfx);
  if (rc != PA_OK) return rc;
  // 3. merge, each row with its own group's parts
  const int* parts = prefill::shared_prefix_split_count(ws + sl.prefix);
  const int* split = prefill::shared_prefix_split_blocks(ws + sl.prefix);
  const int rows = num_seqs * num_q_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (dtype == PA_BF16)
    e = head_dim == 128
            ? cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__nv_bfloat16, 128>, po, plse, parts,
                                 so, slse, static_cast<__nv_bfloat16*>(out), rows, block_tables, 0,
                                 num_seqs, max_blocks_per_seq, status, seq_blocks, split,
                                 num_q_heads)
            : cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__nv_bfloat16, 64>, po, plse, parts,
                                 so, slse, static_cast<__nv_bfloat16*>(out), rows, block_tables, 0,
                                 num_seqs, max_blocks_per_seq, status, seq_blocks, split,
                                 num_q_heads);
  else
    e = head_dim == 128
            ? cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__half, 128>, po, plse, parts, so,
                                 slse, static_cast<__half*>(out), rows, block_tables, 0, num_seqs,
                                 max_blocks_per_seq, status, seq_blocks, split, num_q_heads)
            : cudaLaunchKernelEx(&cfg, cascade_combine_kernel<__half, 64>, po, plse, parts, so,
                                 slse, static_cast<__half*>(out), rows, block_tables, 0, num_seqs,
                                 max_blocks_per_seq, status, seq_blocks, split, num_q_heads);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: merge launch failed: %s", who, cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace

extern "C" {

PA_API int pa_paged_attention_decode_shared_prefix(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int prefix_blocks, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_shared_prefix");
  return shared_prefix_impl(SharedMode::kPlanAndRun, q, k_cache, v_cache, block_tables,
                            context_lens, prefix_blocks, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                            workspace, workspace_bytes, stream,
                            "paged_attention_decode_shared_prefix");
}

PA_API int pa_paged_attention_decode_shared_prefix_plan(
    const int32_t* context_lens, int prefix_blocks, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, float scale, int dtype,
    void* workspace, size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_shared_prefix_plan");
  return shared_prefix_impl(SharedMode::kPlanOnly, nullptr, nullptr, nullptr, nullptr,
                            context_lens, prefix_blocks, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, max_blocks_per_seq, 0, scale, dtype, nullptr, workspace,
                            workspace_bytes, stream, "paged_attention_decode_shared_prefix_plan");
}

PA_API int pa_paged_attention_decode_shared_prefix_run(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int prefix_blocks, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_shared_prefix_run");
  return shared_prefix_impl(SharedMode::kRunOnly, q, k_cache, v_cache, block_tables,
                            context_lens, prefix_blocks, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                            workspace, workspace_bytes, stream,
                            "paged_attention_decode_shared_prefix_run");
}

PA_API int pa_paged_attention_decode_grouped_prefix_workspace_size(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
    size_t* bytes) {
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               PA_BF16, "paged_attention_decode_grouped_prefix_workspace_size");
  if (rc != PA_OK) return rc;
  if (!bytes) return fail(PA_ERR_INVALID_ARG, "grouped_prefix_workspace_size: bytes is NULL");
  *bytes = std::max(
      grouped_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total,
      fused_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total);
  return PA_OK;
}

PA_API int pa_paged_attention_decode_grouped_prefix(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* group_start, const int32_t* group_prefix_blocks,
    int num_groups, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* out, void* workspace,
    size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_grouped_prefix");
  return grouped_prefix_impl(SharedMode::kPlanAndRun, q, k_cache, v_cache, block_tables,
                             context_lens, group_start, group_prefix_blocks, num_groups, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_blocks,
                             scale, dtype, out, workspace, workspace_bytes, stream,
                             "paged_attention_decode_grouped_prefix");
}

PA_API int pa_paged_attention_decode_grouped_prefix_plan(
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* group_start,
    const int32_t* group_prefix_blocks, int num_groups, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, float scale, int dtype,
    void* workspace, size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_grouped_prefix_plan");
  return grouped_prefix_impl(SharedMode::kPlanOnly, nullptr, nullptr, nullptr, block_tables,
                             context_lens, group_start, group_prefix_blocks, num_groups, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, 0, scale,
                             dtype, nullptr, workspace, workspace_bytes, stream,
                             "paged_attention_decode_grouped_prefix_plan");
}

PA_API int pa_paged_attention_decode_grouped_prefix_run(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* group_start, const int32_t* group_prefix_blocks, int num_groups, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
    float scale, int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_grouped_prefix_run");
  return grouped_prefix_impl(SharedMode::kRunOnly, q, k_cache, v_cache, block_tables, nullptr,
                             group_start, group_prefix_blocks, num_groups, num_seqs, num_q_heads,
                             num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype,
                             out, workspace, workspace_bytes, stream,
                             "paged_attention_decode_grouped_prefix_run");
}

PA_API int pa_paged_attention_decode_shared_prefix_append_run(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    int prefix_blocks, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* out, void* workspace,
    size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_shared_prefix_append_run");
  const char* who = "paged_attention_decode_shared_prefix_append_run";
  AppendArgs app;
  int rc = append_args(k_new, v_new, slot_mapping, app, who);
  if (rc != PA_OK) return rc;
  return shared_prefix_impl(SharedMode::kRunOnly, q, k_cache, v_cache, block_tables,
                            context_lens, prefix_blocks, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                            workspace, workspace_bytes, stream, who, app);
}

PA_API int pa_paged_attention_decode_grouped_prefix_append_run(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* group_start,
    const int32_t* group_prefix_blocks, int num_groups, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_decode_grouped_prefix_append_run");
  const char* who = "paged_attention_decode_grouped_prefix_append_run";
  AppendArgs app;
  int rc = append_args(k_new, v_new, slot_mapping, app, who);
  if (rc != PA_OK) return rc;
  return grouped_prefix_impl(SharedMode::kRunOnly, q, k_cache, v_cache, block_tables, nullptr,
                             group_start, group_prefix_blocks, num_groups, num_seqs, num_q_heads,
                             num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype,
                             out, workspace, workspace_bytes, stream, who, app);
}

PA_API int pa_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                     void* out, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  PA_TRACE("pa_paged_attention_decode");
  const char* who = "paged_attention_decode";
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = check_run_args(q, k_cache, v_cache, block_tables, context_lens, out, num_kv_heads,
                      num_blocks, who);
  if (rc != PA_OK) return rc;
  rc = check_workspace(workspace, workspace_bytes,
                       workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                        max_blocks_per_seq),
                       who);
  if (rc != PA_OK) return rc;
  if (dtype != PA_F32) {
    rc = plan_impl(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                   workspace, workspace_bytes, s, who);
    if (rc != PA_OK) return rc;
  }
  return run_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                  workspace, workspace_bytes, s, who);
}

}  // extern "C"

// ====================================================== no-allocation variant
// Some callers cannot hand this library a device workspace: they run inside a
// host framework that owns the whole device-memory budget (a serving engine's
// pre-reserved pool, a process capped at its memory limit) and may not call
// cudaMalloc themselves.  For them the decode path can use a scratch area
// compiled into this library instead: a fixed-size array in device memory
// that every GPU loading the library holds until the process exits.
namespace pa {
namespace decode {
namespace {

constexpr size_t kStaticScratchBytes = size_t(128) << 20;  // 128 MiB per device
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct ScratchSlot {
  std::once_flag once;
  void* addr = nullptr;
  cudaError_t error = cudaSuccess;
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of this device's scratch array (looked up once per device,
// with that device current; the host-side name of the array is not a device
// address).
int static_scratch(void** out) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "paged_attention_decode_noalloc: no current CUDA device");
  ScratchSlot& slot = g_scratch[device];
  std::call_once(slot.once, [&] {
    slot.error = cudaGetSymbolAddress(&slot.addr, g_static_scratch);
    if (slot.error != cudaSuccess) slot.addr = nullptr;
  });
  if (!slot.addr)
    return fail(PA_ERR_CUDA, "paged_attention_decode_noalloc: cudaGetSymbolAddress failed: %s",
                cudaGetErrorString(slot.error));
  *out = slot.addr;
  return PA_OK;
}

}  // namespace
}  // namespace decode
}  // namespace pa

extern "C" {

PA_API int pa_paged_attention_decode_noalloc(const void* q, const void* k_cache,
                                             const void* v_cache, const int32_t* block_tables,
                                             const int32_t* context_lens, int num_seqs,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int max_blocks_per_seq, int num_blocks, float scale,
                                             int dtype, void* out, void* stream) {
  PA_TRACE("pa_paged_attention_decode_noalloc");
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode_noalloc: sizes must be positive");
  if (layout_too_large(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq))
    return fail(PA_ERR_INVALID_ARG,
                "paged_attention_decode_noalloc: these shapes need far more than the library's "
                "built-in scratch of %zu bytes",
                kStaticScratchBytes);
  const size_t need =
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total;
  if (need > kStaticScratchBytes)
    return fail(PA_ERR_INVALID_ARG,
                "paged_attention_decode_noalloc: these shapes need %zu bytes of scratch, more than "
                "the %zu built into the library; pass a workspace to pa_paged_attention_decode",
                need, kStaticScratchBytes);
  if (num_seqs == 0) return PA_OK;
  void* scratch = nullptr;
  const int rc = static_scratch(&scratch);
  if (rc != PA_OK) return rc;
  return pa_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                   num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                   num_blocks, scale, dtype, out, scratch, kStaticScratchBytes,
                                   stream);
}

}  // extern "C"
