// Chunked-prefill attention over the paged KV cache, for sm_103a.
//
// What it computes: sequence b holds context_lens[b] tokens; its newest T_b of
// them (a prefill chunk, K/V already stored in the cache) have query rows
// query_start[b] .. query_start[b + 1] - 1.  Query row i (token position
// p = context_lens[b] - T_b + i) of query head h attends over tokens 0 .. p:
//   out[row][h] = softmax_t(scale * q[row][h] . K_t) . V_t,   t <= p,
// K_t / V_t read through the block table (KV head h / G).  OS-lab appendix
// "Lazy Allocation 与 Copy-on-Write 在 LLM 推理系统中的应用", section 2.1
// (prefill writes the K/V of every prompt token to the cache); "vLLM: treating
// the KV cache as virtual memory", section "KV 的体积从哪来，页表如何把它切开"
// (chunked prefill cuts a long prompt into pieces run between decode steps).
// Decode is the case T_b = 1.
//
// Design (ours; the pages give no kernel):
//  * A work item is (sequence, KV head, block of 64 query rows, KV split).  A
//    query row is one (token, query head of the group) pair, so one item's
//    rows are up to 64 / G tokens of the chunk times the G heads that share
//    the KV head: every K/V tile is read once for all of them.
//  * plan kernel (1 CTA): query blocks per sequence, the KV range each needs
//    (causal: up to its last token), KV splits only when the query blocks
//    alone cannot fill the GPU, units ordered by size (largest first).
//  * attention kernel: persistent CTAs of 4 warps, 16 query rows each, sharing
//    a TMA-fed ring of 16-token K/V blocks (one issuing thread; a stage is
//    refilled once all 4 warps have released it).  Per block and warp:
//    S = Q K^T (16 rows x 16 tokens, m16n8k16 on the tensor cores), causal
//    and context masks, online softmax in base 2, P reused in registers as
//    the A operand of O += P V (V^T fragments via ldmatrix.trans).  Splits of
//    a query block are merged with log-sum-exp weights by the CTA that
//    finishes the last one.
//  * fp32 caches take a plain CUDA-core path (one warp per (row, head)).
//  * Every wait is an mbarrier or spin wait with a time limit; running out
//    sets the timeout bit of the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "trace.h"
#include "pagedattn.h"
#include "prefill.h"
#include "tc05.cuh"
#include "status.h"
#include "tensor_map.h"

namespace pa {
namespace prefill {

constexpr int kBlockSize = 16;       // tokens per physical block
constexpr int kWarps = 4;            // math warps per CTA
constexpr int kRows = kWarps * 16;   // query rows per work item
constexpr int kStages = 4;           // depth of the CTA's K/V ring
constexpr int kMaxGroup = 8;         // query heads per KV head
constexpr int kMinSplitBlocks = 16;  // smallest KV split
constexpr int kPartialItems = 1024;  // (split unit, KV head) partial results, at most
constexpr int kSizeBuckets = 32;     // work-list order: floor(log2(blocks)) buckets
constexpr int kMaxSplits = 64;       // splits of one query block (the merge's weights fit the ring)

// Splits of a query block of nb KV blocks at split size `split` (0: none).
__host__ __device__ __forceinline__ int nsplits_of(int nb, int split) {
  if (!split) return 1;
  const int ns = (nb + split - 1) / split;
  return ns < kMaxSplits ? ns : kMaxSplits;
}

// Workspace header words.
constexpr int kHdrNext = 0, kHdrTotal = 1, kHdrDone = 2, kHdrSignature = 3;
// shared-prefix mode: how many (o, lse) parts per row the phase left in
// cas_o / cas_lse for the caller to merge (1 when it merged them itself);
// the split size in blocks behind it (0: none, or merged in-kernel), from
// which the caller works out each group's count in grouped mode
constexpr int kHdrSplits = 4, kHdrSplitBlocks = 5;

struct Params {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  int num_seqs, total_q, num_q_heads, num_kv_heads, group, head_dim;
  int max_blocks, num_blocks;
  int ncta;          // CTAs the attention kernel runs with (plan: how much to split)
  int units_cap;     // unit slots in the workspace
  int partial_cap;   // partial-result units in the workspace (per KV head)
  int signature;
  // Shared-prefix mode (shared_ctx > 0): the batch's decode queries are the
  // total_q "tokens" of one sequence (num_seqs = 1) whose K/V are the
  // shared_ctx tokens of the shared prefix (block_tables row 0); every row
  // attends all of them (no causal mask), and the results go to cas_o /
  // cas_lse (fp32 o and base-2 log-sum-exp per (row, head)) instead of out.
  int shared_ctx;
  // Grouped shared-prefix mode (shared_blocks non-null): num_seqs groups of
  // decode queries, group g the rows query_start[g] .. query_start[g + 1] - 1
  // (one per sequence, so the group's first member has table row
  // query_start[g]), attending the group's own prefix of shared_blocks[g]
  // blocks (no causal mask); results as in shared-prefix mode.
  const int32_t* shared_blocks;
  int no_split;      // plan: never split a unit's KV range (tcgen05 kernel)
  // shared-prefix mode on the tcgen05 kernel: split s of every row writes its
  // own (o, lse) to slot s of cas_o / cas_lse ([kSharedMaxSplits][rows]...);
  // the caller merges them (the split count is header word kHdrSplits)
  int defer_merge;
  float* cas_o;      // [total_q * num_q_heads][head_dim]
  float* cas_lse;    // [total_q * num_q_heads]
  // tcgen05 kernel: whole warps of output rows go out through the tensor
  // map of out (tensor-copy stores from shared memory), else thread by thread
  int out_tma;
  float scale, scale_log2;
  int* header;
  int4* units;       // 2 x int4 per unit (see plan)
  int* arrivals;     // [partial_cap][num_kv_heads]
  float* part_lse;   // [partial_cap][num_kv_heads][kRows]
  float* part_o;     // [partial_cap][num_kv_heads][kRows][head_dim]
  unsigned* status;
  unsigned long long timeout_ns;
};

struct Layout {
  size_t header, units, arrivals, part_lse, part_o, total;
  int units_cap, partial_cap;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline Layout workspace_layout(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                               int head_dim) {
  Layout l;
  const int group = num_q_heads / num_kv_heads;
  // query blocks: sum over sequences of ceil(T_b G / 64) <= total_q G / 64 + num_seqs
  const long long qblocks = (long long)total_q * group / kRows + num_seqs + 1;
  l.partial_cap = std::max(1, kPartialItems / num_kv_heads);
  l.units_cap = int(std::min<long long>(qblocks + l.partial_cap, 1ll << 30));
  l.header = 0;
  l.units = align256(256);
  l.arrivals = align256(l.units + size_t(l.units_cap) * 32);
  l.part_lse = align256(l.arrivals + size_t(l.partial_cap) * num_kv_heads * 4);
  l.part_o = align256(l.part_lse + size_t(l.partial_cap) * num_kv_heads * kRows * 4);
  l.total = align256(l.part_o + size_t(l.partial_cap) * num_kv_heads * kRows * head_dim * 4);
  return l;
}

inline int signature_of(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                        int head_dim, int max_blocks) {
  uint32_t h = 2166136261u;
  const int v[7] = {num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, max_blocks, 0x5EED};
  for (int x : v) {
    h ^= uint32_t(x);
    h *= 16777619u;
  }
  return int(h | 1u);
}

// ------------------------------------------------------------------ plan
// A query block qb of sequence b covers rows qb*64 .. of the sequence's
// T_b * G rows; its last row's token sits at position ctx - T_b + i_last,
// so it needs KV blocks 0 .. that position / 16.
template <int ROWS = kRows>
__device__ __forceinline__ int qblock_blocks(int ctx, int qlen, int group, int qb,
                                             bool all_tokens = false) {
  if (all_tokens) return (ctx + kBlockSize - 1) / kBlockSize;
  const int rows = qlen * group;
  const int last_row = min((qb + 1) * ROWS, rows) - 1;
  const int pos = ctx - qlen + last_row / group;
  return pos / kBlockSize + 1;
}

__device__ __forceinline__ int size_bucket(int n) { return 31 - __clz(n); }  // floor(log2 n)

constexpr int kPlanThreads = 256;

// ROWS: query rows per unit (64 for the mma.sync kernel, 128 for the
// tcgen05 one, which never splits: p.no_split).
template <int ROWS>
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const Params p) {
  __shared__ unsigned long long s_blocks;
  __shared__ int s_qblocks, s_split_units, s_split, s_slot, s_group, s_maxnb;
  __shared__ int hist[kSizeBuckets];
  __shared__ int bucket[kSizeBuckets];
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();  // the previous kernel may still read the workspace
  const int tid = threadIdx.x;
  const int G = p.group;
  const int cap = p.max_blocks * kBlockSize;
  if (tid == 0) {
    s_blocks = 0;
    s_qblocks = 0;
    s_slot = 0;
    s_group = 0;
    s_maxnb = 0;
  }
  if (tid < kSizeBuckets) hist[tid] = 0;
  __syncthreads();

  // a sequence's chunk: (ctx, qlen), or qlen = 0 when its lengths are invalid
  const bool shared = p.shared_ctx > 0 || p.shared_blocks;
  auto chunk = [&](int b, int& ctx, int& qlen) {
    if (p.shared_blocks) {  // group b: its rows over its own prefix
      const int nb = p.shared_blocks[b];
      const int q0 = p.query_start[b], q1 = p.query_start[b + 1];
      ctx = nb * kBlockSize;
      qlen = q1 - q0;
      if (nb < 0 || ctx > cap || qlen < 0 || q0 < 0 || q1 > p.total_q) {
        dev::flag_status(p.status, kStatusBounds);
        qlen = 0;
      }
      if (ctx <= 0) qlen = 0;
      return;
    }
    if (shared) {
      ctx = p.shared_ctx <= cap ? p.shared_ctx : 0;
      qlen = ctx > 0 ? p.total_q : 0;
      return;
    }
    ctx = p.context_lens[b];
    const int q0 = p.query_start[b], q1 = p.query_start[b + 1];
    qlen = q1 - q0;
    if (ctx < 0 || ctx > cap || qlen < 0 || qlen > ctx || q0 < 0 || q1 > p.total_q) {
      dev::flag_status(p.status, kStatusBounds);
      qlen = 0;
    }
  };

  // pass 1: query blocks and KV blocks in all
  for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
    int ctx, qlen;
    chunk(b, ctx, qlen);
    const int nq = (qlen * G + ROWS - 1) / ROWS;
    unsigned long long blocks = 0;
    for (int qb = 0; qb < nq; ++qb) blocks += qblock_blocks<ROWS>(ctx, qlen, G, qb, shared);
    if (nq) {
      atomicAdd(&s_qblocks, nq);
      atomicAdd(&s_blocks, blocks);
      if (shared) atomicMax(&s_maxnb, (ctx + kBlockSize - 1) / kBlockSize);
    }
  }
  __syncthreads();
  // Split size: none while the query blocks alone give every CTA two items;
  // otherwise aim at three items per CTA, never below kMinSplitBlocks, and
  // double it until the split units fit the workspace's partial results.
  if (tid == 0 && s_qblocks > p.units_cap - p.partial_cap) {
    // inconsistent query_start (overlapping chunks): more query blocks than
    // total_q can give; refuse the whole batch
    dev::flag_status(p.status, kStatusBounds);
    s_qblocks = 0;
  }
  __syncthreads();
  if (s_qblocks == 0) {
    if (tid == 0) {
      p.header[kHdrTotal] = 0;
      p.header[kHdrNext] = 0;
      p.header[kHdrDone] = 0;
      p.header[kHdrSplits] = 1;
      p.header[kHdrSplitBlocks] = 0;
      p.header[kHdrSignature] = p.signature;
    }
    return;
  }
  if (tid == 0) {
    const long long items = (long long)s_qblocks * p.num_kv_heads;
    int split = 0;
    if (!p.no_split && items < 2ll * p.ncta && s_qblocks > 0) {
      const long long want = (long long)s_blocks * p.num_kv_heads / (3ll * p.ncta) + 1;
      // the shared-prefix phase has few, short rows: allow shorter splits
      split = int(std::max<long long>(shared ? kMinSplitBlocks / 2 : kMinSplitBlocks, want));
      // parts left for the caller: at most kSharedMaxSplits per row (the
      // longest prefix decides)
      if (p.defer_merge) split = std::max(split, (s_maxnb + kSharedMaxSplits - 1) / kSharedMaxSplits);
    }
    s_split = split;
  }
  __syncthreads();
  for (int round = 0; round < 24 && s_split > 0; ++round) {
    if (tid == 0) s_split_units = 0;
    __syncthreads();
    const int split = s_split;
    for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
      int ctx, qlen;
      chunk(b, ctx, qlen);
      const int nq = (qlen * G + ROWS - 1) / ROWS;
      int units = 0;
      for (int qb = 0; qb < nq; ++qb) {
        const int ns = nsplits_of(qblock_blocks<ROWS>(ctx, qlen, G, qb, shared), split);
        if (ns > 1 && !p.defer_merge) units += ns * (ROWS / kRows);  // partial slots of kRows rows
      }
      if (units) atomicAdd(&s_split_units, units);
    }
    __syncthreads();
    if (tid == 0) {
      if (s_split_units > p.partial_cap) s_split = s_split > (1 << 24) ? 0 : s_split * 2;
      else s_split = -s_split;  // fits: stop (sign marks "done")
    }
    __syncthreads();
    if (s_split <= 0) break;
  }
  __syncthreads();
  const int split = s_split < 0 ? -s_split : 0;  // 0: no splitting

  // pass 2: the work list is ordered by size, largest first, at the grain
  // of sequences: all of a sequence's units go into the size bucket of its
  // largest one, next to each other, so the query blocks of a (sequence, KV
  // head) run at about the same time on different SMs and read its K/V
  // tiles while they are in L2.  (A query block's splits are balanced.)
  auto units_of = [&](int b, int& count, int& largest) {
    int ctx, qlen;
    chunk(b, ctx, qlen);
    const int nq = (qlen * G + ROWS - 1) / ROWS;
    count = 0;
    largest = 0;
    for (int qb = 0; qb < nq; ++qb) {
      const int nb = qblock_blocks<ROWS>(ctx, qlen, G, qb, shared);
      const int ns = nsplits_of(nb, split);
      count += ns;
      largest = max(largest, (nb + ns - 1) / ns);
    }
  };
  for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
    int count, largest;
    units_of(b, count, largest);
    if (count) atomicAdd(&hist[size_bucket(largest)], count);
  }
  __syncthreads();
  if (tid == 0) {
    int pos = 0;
    for (int r = kSizeBuckets - 1; r >= 0; --r) {
      bucket[r] = pos;
      pos += hist[r];
    }
    p.header[kHdrTotal] = pos * p.num_kv_heads;
    p.header[kHdrNext] = 0;
    p.header[kHdrDone] = 0;
    p.header[kHdrSplits] = p.defer_merge && shared ? nsplits_of(s_maxnb, split) : 1;
    p.header[kHdrSplitBlocks] = p.defer_merge && shared ? split : 0;
    p.header[kHdrSignature] = p.signature;
  }
  __syncthreads();
  // pass 3: place the units (the last query block, the largest, first),
  // claim partial slots and arrival counters for the split ones.  Unit =
  // {b, qb, first block, blocks} {split << 16 | nsplit, first partial slot,
  // arrival group, ctx}.
  for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
    int count, largest;
    units_of(b, count, largest);
    if (count == 0) continue;
    int pos = atomicAdd(&bucket[size_bucket(largest)], count);
    int ctx, qlen;
    chunk(b, ctx, qlen);
    const int nq = (qlen * G + ROWS - 1) / ROWS;
    for (int qb = nq - 1; qb >= 0; --qb) {
      const int nb = qblock_blocks<ROWS>(ctx, qlen, G, qb, shared);
      const int ns = nsplits_of(nb, split);
      const int base = nb / ns, big = nb - base * ns;
      int slot = -1, grp = -1;
      if (ns > 1 && !p.defer_merge) {
        slot = atomicAdd(&s_slot, ns * (ROWS / kRows));
        grp = atomicAdd(&s_group, 1);
        for (int g = 0; g < p.num_kv_heads; ++g) p.arrivals[size_t(grp) * p.num_kv_heads + g] = 0;
      }
      int first = 0;
      for (int s = 0; s < ns; ++s) {
        const int n = s < big ? base + 1 : base;
        p.units[2 * pos] = make_int4(b, qb, first, n);
        p.units[2 * pos + 1] = make_int4((s << 16) | ns, slot, grp, ctx);
        ++pos;
        first += n;
      }
    }
  }
}

// --------------------------------------------------------- tensor-core path
template <int D>
struct Smem {
  static constexpr int kTileBytes = kBlockSize * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr size_t kBytes =
      1024 /* alignment slack */ + size_t(kStages) * kStageBytes + 2 * kStages * 8 + 64;
};

// One work item as every thread of the CTA holds it.
struct Item {
  int b, qb, first, nblk, s, ns, slot, grp, ctx, g;
  int q_first, qlen;
};

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32, 3)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  using S = Smem<D>;
  using M = dev::Mma<T>;
  constexpr int KT = D / 16;      // 16-wide steps along head_dim
  constexpr int ND = D / 8;       // 8-wide output column tiles
  constexpr int HALVES = D / 64;  // 128-byte TMA boxes per tile row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + size_t(kStages) * S::kStageBytes);
  uint64_t* empty = full + kStages;
  int* s_claim = reinterpret_cast<int*>(empty + kStages);
  int* s_last = s_claim + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;  // fragment row group / column pair
  const bool producer = threadIdx.x == 0;
  if (producer) {
    for (int i = 0; i < kStages; ++i) {
      dev::mbar_init(&full[i], 1);
      dev::mbar_init(&empty[i], kWarps);
    }
    dev::mbar_fence_init();
    dev::prefetch_tensormap(&tmap_k);
    dev::prefetch_tensormap(&tmap_v);
  }
  __syncthreads();
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();

  const unsigned long long tmo = p.timeout_ns;
  const int G = p.group, Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const bool shared = p.shared_ctx > 0 || p.shared_blocks;
  const bool planned = *reinterpret_cast<volatile int*>(&p.header[kHdrSignature]) == p.signature;
  if (!planned && blockIdx.x == 0 && threadIdx.x == 0) dev::flag_status(p.status, kStatusPlan);
  const int total = planned ? *reinterpret_cast<volatile int*>(&p.header[kHdrTotal]) : 0;
  const uint64_t policy = dev::l2_policy_evict_first();
  int kc = 0;  // blocks consumed by this warp so far (same for every warp)
  int ik = 0;  // blocks issued so far (producer only)
  bool ok = true;

  // Warp 0 issues the ring's copies; its lane l holds table entry tbl_base + l
  // of the current item (refreshed every 32 blocks), so no copy waits on a
  // dependent table read.
  int tbl = 0, tbl_base = -32;
  // Issues block k (the item's block j) into the ring, once the stage's
  // previous block has been released by every warp.  Called by all of warp 0.
  auto issue = [&](const Item& it, int j, int k) -> bool {
    if ((j & ~31) != tbl_base) {
      tbl_base = j & ~31;
      tbl = tbl_base + lane < it.nblk
                ? p.block_tables[size_t(shared ? it.q_first : it.b) * p.max_blocks + it.first +
                                 tbl_base + lane]
                : 0;
      if (tbl < 0 || tbl >= p.num_blocks) {
        dev::flag_status(p.status, kStatusBounds);
        tbl = 0;
      }
    }
    const int phys = __shfl_sync(0xffffffffu, tbl, j & 31);
    const int st = k % kStages;
    bool ok_ = true;
    if (lane == 0) {
      if (k >= kStages &&
          !dev::mbar_wait_bounded(&empty[st], ((k / kStages) - 1) & 1, tmo, p.status)) {
        ok_ = false;
      } else {
        dev::mbar_arrive_expect_tx(&full[st], S::kStageBytes);
        uint8_t* dst = ring + size_t(st) * S::kStageBytes;
        const int y = (phys * Hkv + it.g) * kBlockSize;
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
          dev::tma_load_2d(dst + h * 2048, &tmap_k, h * 64, y, &full[st], policy);
          dev::tma_load_2d(dst + S::kTileBytes + h * 2048, &tmap_v, h * 64, y, &full[st], policy);
        }
      }
    }
    return __shfl_sync(0xffffffffu, ok_, 0);
  };

  bool first_claim = true;
  for (;;) {
    if (producer) {
      // the first item of every CTA is dealt statically, the rest come from
      // the counter
      *s_claim = first_claim ? int(blockIdx.x)
                             : int(gridDim.x) + atomicAdd(&p.header[kHdrNext], 1);
    }
    first_claim = false;
    __syncthreads();
    const int x = *s_claim;
    __syncthreads();
    if (x >= total) break;
    Item it;
    {
      const int4 u0 = p.units[2 * (x / Hkv)], u1 = p.units[2 * (x / Hkv) + 1];
      it.g = x % Hkv;
      it.b = u0.x;
      it.qb = u0.y;
      it.first = u0.z;
      it.nblk = u0.w;
      it.s = u1.x >> 16;
      it.ns = u1.x & 0xffff;
      it.slot = u1.y;
      it.grp = u1.z;
      it.ctx = u1.w;
      // shared-prefix mode: the batch's queries are the rows of one sequence
      // (grouped: the group's rows)
      const bool starts = !shared || p.shared_blocks;
      it.q_first = starts ? p.query_start[it.b] : 0;
      it.qlen = starts ? p.query_start[it.b + 1] - it.q_first : p.total_q;
    }
    // the ring's first blocks of this item
    tbl_base = -32;
    if (warp == 0) {
      for (int j = 0; j < it.nblk && j < kStages; ++j, ++ik)
        if (!issue(it, j, ik)) ok = false;
    }

    // ---- this warp's 16 query rows: ra = gq, rb = gq + 8 (of the warp's 16)
    const int row0 = it.qb * kRows + warp * 16;  // first row among (b, g)'s T * G rows
    const int nrows = it.qlen * G;
    const int ra = row0 + gq, rb = ra + 8;
    const bool va = ra < nrows, vb = rb < nrows;
    const int pos_a = va ? (shared ? it.ctx - 1 : it.ctx - it.qlen + ra / G) : -1;
    const int pos_b = vb ? (shared ? it.ctx - 1 : it.ctx - it.qlen + rb / G) : -1;
    const T* qa = static_cast<const T*>(p.q) +
                  (size_t(it.q_first + (va ? ra / G : 0)) * Hq + it.g * G + (va ? ra % G : 0)) * D;
    const T* qbp = static_cast<const T*>(p.q) +
                   (size_t(it.q_first + (vb ? rb / G : 0)) * Hq + it.g * G + (vb ? rb % G : 0)) * D;
    uint32_t qf[KT][4];
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const int c = 16 * kk + 2 * tq;
      qf[kk][0] = va ? *reinterpret_cast<const uint32_t*>(qa + c) : 0u;
      qf[kk][1] = vb ? *reinterpret_cast<const uint32_t*>(qbp + c) : 0u;
      qf[kk][2] = va ? *reinterpret_cast<const uint32_t*>(qa + c + 8) : 0u;
      qf[kk][3] = vb ? *reinterpret_cast<const uint32_t*>(qbp + c + 8) : 0u;
    }
    float o[ND][4];
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    const float sl2 = p.scale_log2;

    for (int j = 0; j < it.nblk; ++j, ++kc) {
      const int st = kc % kStages;
      if (!dev::mbar_wait_bounded(&full[st], (kc / kStages) & 1, tmo, p.status)) {
        ok = false;
        break;
      }
      const uint32_t kt = dev::smem_u32(ring + size_t(st) * S::kStageBytes);
      const uint32_t vt = kt + S::kTileBytes;
      const int t0 = (it.first + j) * kBlockSize;  // first token of the block
      // ---- S = Q K^T: 16 rows x 16 tokens (two 8-token column tiles)
      // two accumulation chains per column tile (even / odd k-steps) halve
      // the dependent MMA latency
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
        const int mi = lane >> 3;
        const int tok = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          const int gc = 2 * kk + (mi & 1);
          const uint32_t addr =
              kt + (gc >> 3) * 2048 + tok * 128 + ((((gc & 7) ^ (tok & 7))) << 4);
          uint32_t b0, b1, b2, b3;
          dev::ldmatrix_x4(addr, b0, b1, b2, b3);
          M::run(kk & 1 ? e0 : s0, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          M::run(kk & 1 ? e1 : s1, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s0[i] += e0[i];
          s1[i] += e1[i];
        }
      }
      // ---- causal / context mask, base-2 scores
      const int c0 = t0 + 2 * tq, c1 = c0 + 8;  // tokens of s0[0], s1[0]
      float xa[4], xb[4];
      xa[0] = c0 <= pos_a ? s0[0] * sl2 : -INFINITY;
      xa[1] = c0 + 1 <= pos_a ? s0[1] * sl2 : -INFINITY;
      xa[2] = c1 <= pos_a ? s1[0] * sl2 : -INFINITY;
      xa[3] = c1 + 1 <= pos_a ? s1[1] * sl2 : -INFINITY;
      xb[0] = c0 <= pos_b ? s0[2] * sl2 : -INFINITY;
      xb[1] = c0 + 1 <= pos_b ? s0[3] * sl2 : -INFINITY;
      xb[2] = c1 <= pos_b ? s1[2] * sl2 : -INFINITY;
      xb[3] = c1 + 1 <= pos_b ? s1[3] * sl2 : -INFINITY;
      float bma = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
      float bmb = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
      bma = fmaxf(bma, __shfl_xor_sync(0xffffffffu, bma, 1));
      bma = fmaxf(bma, __shfl_xor_sync(0xffffffffu, bma, 2));
      bmb = fmaxf(bmb, __shfl_xor_sync(0xffffffffu, bmb, 1));
      bmb = fmaxf(bmb, __shfl_xor_sync(0xffffffffu, bmb, 2));
      const float mna = fmaxf(ma, bma), mnb = fmaxf(mb, bmb);
      // a row with nothing unmasked yet keeps m = -inf: use 0 as its reference
      const float ra0 = mna == -INFINITY ? 0.f : mna, rb0 = mnb == -INFINITY ? 0.f : mnb;
      const float ala = dev::fast_exp2(ma - ra0), alb = dev::fast_exp2(mb - rb0);
      ma = mna;
      mb = mnb;
      const uint32_t pa01 = M::pack(dev::fast_exp2(xa[0] - ra0), dev::fast_exp2(xa[1] - ra0));
      const uint32_t pb01 = M::pack(dev::fast_exp2(xb[0] - rb0), dev::fast_exp2(xb[1] - rb0));
      const uint32_t pa23 = M::pack(dev::fast_exp2(xa[2] - ra0), dev::fast_exp2(xa[3] - ra0));
      const uint32_t pb23 = M::pack(dev::fast_exp2(xb[2] - rb0), dev::fast_exp2(xb[3] - rb0));
      {
        const float2 f0 = M::unpack(pa01), f1 = M::unpack(pa23);
        const float2 g0 = M::unpack(pb01), g1 = M::unpack(pb23);
        la = la * ala + (f0.x + f0.y + f1.x + f1.y);
        lb = lb * alb + (g0.x + g0.y + g1.x + g1.y);
      }
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        o[nd][0] *= ala;
        o[nd][1] *= ala;
        o[nd][2] *= alb;
        o[nd][3] *= alb;
      }
      // ---- O += P V: P (16 rows x 16 tokens) is the A operand as computed
      {
        const int mi = lane >> 3;
        const int tok = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
        for (int nd = 0; nd < ND; nd += 2) {
          const int gc = nd + (mi >> 1);  // 16-byte chunk = 8 columns
          const uint32_t addr =
              vt + (gc >> 3) * 2048 + tok * 128 + ((((gc & 7) ^ (tok & 7))) << 4);
          uint32_t b0, b1, b2, b3;
          dev::ldmatrix_x4_trans(addr, b0, b1, b2, b3);
          M::run(o[nd], pa01, pb01, pa23, pb23, b0, b1);
          M::run(o[nd + 1], pa01, pb01, pa23, pb23, b2, b3);
        }
      }
      // the stage is read: order those reads before the copy that reuses it
      dev::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&empty[st]);
      if (warp == 0 && j + kStages < it.nblk) {
        if (!issue(it, j + kStages, ik)) ok = false;
        ++ik;
      }
    }
    // every thread agrees before anyone leaves the loop (no one may be left
    // waiting at a CTA barrier)
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }

    // ---- end of the item: row sums across the quad, then out or partials
    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    const float ia = la > 0.f ? 1.f / la : 0.f, ib = lb > 0.f ? 1.f / lb : 0.f;
    if (it.ns == 1 && shared) {
      // (row, head) index of the rows: token ra / G is the batch's sequence
      const size_t ha = size_t(it.q_first + (va ? ra / G : 0)) * Hq + it.g * G + (va ? ra % G : 0);
      const size_t hb = size_t(it.q_first + (vb ? rb / G : 0)) * Hq + it.g * G + (vb ? rb % G : 0);
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const int c = nd * 8 + 2 * tq;
        if (va) *reinterpret_cast<float2*>(p.cas_o + ha * D + c) = make_float2(o[nd][0] * ia, o[nd][1] * ia);
        if (vb) *reinterpret_cast<float2*>(p.cas_o + hb * D + c) = make_float2(o[nd][2] * ib, o[nd][3] * ib);
      }
      if (tq == 0) {
        if (va) p.cas_lse[ha] = la > 0.f ? ma + log2f(la) : -INFINITY;
        if (vb) p.cas_lse[hb] = lb > 0.f ? mb + log2f(lb) : -INFINITY;
      }
    } else if (it.ns == 1) {
      T* oa = static_cast<T*>(p.out) +
              (size_t(it.q_first + (va ? ra / G : 0)) * Hq + it.g * G + (va ? ra % G : 0)) * D;
      T* ob = static_cast<T*>(p.out) +
              (size_t(it.q_first + (vb ? rb / G : 0)) * Hq + it.g * G + (vb ? rb % G : 0)) * D;
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const int c = nd * 8 + 2 * tq;
        if (va) *reinterpret_cast<uint32_t*>(oa + c) = M::pack(o[nd][0] * ia, o[nd][1] * ia);
        if (vb) *reinterpret_cast<uint32_t*>(ob + c) = M::pack(o[nd][2] * ib, o[nd][3] * ib);
      }
    } else {
      const size_t base = (size_t(it.slot + it.s) * Hkv + it.g) * kRows + warp * 16;
      float* pa = p.part_o + (base + gq) * D;
      float* pb = p.part_o + (base + gq + 8) * D;
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const int c = nd * 8 + 2 * tq;
        *reinterpret_cast<float2*>(pa + c) = make_float2(o[nd][0] * ia, o[nd][1] * ia);
        *reinterpret_cast<float2*>(pb + c) = make_float2(o[nd][2] * ib, o[nd][3] * ib);
      }
      if (tq == 0) {
        p.part_lse[base + gq] = la > 0.f ? ma + log2f(la) : -INFINITY;
        p.part_lse[base + gq + 8] = lb > 0.f ? mb + log2f(lb) : -INFINITY;
      }
      // publish (every warp's rows), count; the CTA completing (group, g) merges
      __syncthreads();
      if (producer)
        *s_last = dev::atom_add_acq_rel_gpu(&p.arrivals[size_t(it.grp) * Hkv + it.g], 1) ==
                  it.ns - 1;
      __syncthreads();
      if (*s_last) {
        // The whole CTA merges the item's 64 rows.  Pass 1: one thread per row
        // turns the splits' lse into weights, kept in the (now idle) ring.
        float* wsm = reinterpret_cast<float*>(ring);  // [ns][kRows]
        const size_t sbase = (size_t(it.slot) * Hkv + it.g) * kRows;  // split s adds s*Hkv*kRows
        const size_t sstride = size_t(Hkv) * kRows;
        if (threadIdx.x < kRows) {
          const int r = threadIdx.x;
          float mx = -INFINITY;
          for (int sp = 0; sp < it.ns; ++sp)
            mx = fmaxf(mx, __ldcg(&p.part_lse[sbase + sp * sstride + r]));
          float sum = 0.f;
          for (int sp = 0; sp < it.ns; ++sp) {
            const float x = __ldcg(&p.part_lse[sbase + sp * sstride + r]);
            const float w = x == -INFINITY ? 0.f : dev::fast_exp2(x - mx);
            wsm[sp * kRows + r] = w;
            sum += w;
          }
          const float inv = sum > 0.f ? 1.f / sum : 0.f;
          for (int sp = 0; sp < it.ns; ++sp) wsm[sp * kRows + r] *= inv;
          const int row = it.qb * kRows + r;
          if (shared && row < nrows)
            p.cas_lse[size_t(it.q_first + row / G) * Hq + it.g * G + row % G] =
                sum > 0.f ? mx + log2f(sum) : -INFINITY;
        }
        __syncthreads();
        // Pass 2: thread t owns float4 column t % C4 of rows t / C4 + k * RS;
        // every split's loads for all its rows are in flight together.
        constexpr int C4 = D / 4, RS = kWarps * 32 / C4, NR = kRows / RS;
        const int c4 = threadIdx.x % C4, r0 = threadIdx.x / C4;
        float4 acc[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < it.ns; ++sp) {
          const float4* src = reinterpret_cast<const float4*>(p.part_o + (sbase + sp * sstride) * D);
#pragma unroll
          for (int k = 0; k < NR; ++k) {
            const int r = r0 + k * RS;
            const float w = wsm[sp * kRows + r];
            const float4 v = __ldcg(src + size_t(r) * C4 + c4);
            acc[k].x += w * v.x;
            acc[k].y += w * v.y;
            acc[k].z += w * v.z;
            acc[k].w += w * v.w;
          }
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
          const int row = it.qb * kRows + r0 + k * RS;
          if (row >= nrows) continue;
          const size_t hrow = size_t(it.q_first + row / G) * Hq + it.g * G + row % G;
          if (shared) {
            reinterpret_cast<float4*>(p.cas_o + hrow * D)[c4] = acc[k];
          } else {
            uint2 pk;
            pk.x = M::pack(acc[k].x, acc[k].y);
            pk.y = M::pack(acc[k].z, acc[k].w);
            reinterpret_cast<uint2*>(static_cast<T*>(p.out) + hrow * D)[c4] = pk;
          }
        }
        // the ring is a copy target again after this
        dev::fence_proxy_async_smem();
        __syncthreads();
        if (producer) p.arrivals[size_t(it.grp) * Hkv + it.g] = 0;  // ready for the next run
      }
    }
  }
  if (!ok) {
    // a wait ran out: let this CTA's copies in flight land, then give up
    if (producer)
      for (int k = kc; k < ik; ++k)
        dev::mbar_wait_bounded(&full[k % kStages], (k / kStages) & 1, tmo, p.status);
    return;
  }
  // the last CTA to finish returns the counters to zero
  __syncthreads();
  if (producer && planned) {
    __threadfence();
    if (atomicAdd(&p.header[kHdrDone], 1) == int(gridDim.x) - 1) {
      atomicExch(&p.header[kHdrNext], 0);
      atomicExch(&p.header[kHdrDone], 0);
    }
  }
}

// ------------------------------------------------------- tcgen05 path (d = 128)
// A work item is 256 query rows (rows = tokens x the group's heads, as above)
// of one (sequence, KV head): two 128-row query tiles that share every KV
// tile of the item's causal range, streamed in tiles of 128 tokens (8 paged
// blocks).  Warp roles:
//   warp 8       producer: claims items (two-slot queue), TMA copies of the
//                query tiles and the K / V tiles (separate 2-stage rings)
//   warp 9       one thread issues the 5th-generation tensor-core MMAs
//                  S_w  = Q_w K^T   (M 128, N 128 tokens, K 128; fp32 in TMEM)
//                  O_w += P_w V     (M 128, N 128 = head_dim, K 128 tokens)
//   warps 0-3, 4-7  softmax of query tile 0 / 1, one thread per row (its TMEM
//                lane); while one group works on its scores the tensor core
//                runs the other group's MMAs.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, 128 columns each.  P_w is written
// in the input type over the first 64 columns of S_w and is the A operand of
// O_w += P_w V straight from TMEM; V is the N-contiguous B operand, K the
// K-major B operand of S, as the TMA tiles land.  The softmax exponentiates
// in base 2 against a reference that moves only when a row's maximum grows by
// more than 2^8 (O_w is then rescaled in TMEM; the result is the same either
// way).
// Optional per-role wait counters (SM cycles), compiled in only with
// -DPA_PROFILE_TIMES (a separate build; the default build has none of it).
// Per CTA 32 slots of 8: MMA thread, softmax group 0 (its thread 0), group 1,
// producer lane 0; the last slot of each is the role's total (the meaning of
// each other slot is where it is added).
#ifdef PA_PROFILE_TIMES
__device__ unsigned long long g_pf_times[2048 * 32];
#define PF_DECL long long pf_[8] = {0, 0, 0, 0, 0, 0, 0, 0}; const long long pf_start_ = clock64()
#define PF_WAIT(slot, call)                    \
  ([&]() {                                     \
    const long long t_ = clock64();            \
    const bool r_ = (call);                    \
    pf_[slot] += clock64() - t_;               \
    return r_;                                 \
  }())
#define PF_MARK(name) const long long name = clock64()
#define PF_ADD(slot, since) pf_[slot] += clock64() - (since)
__device__ unsigned long long g_pf_stamps[2048 * 4];
#define PF_STAMP(i)                                                                    \
  do {                                                                                 \
    if (threadIdx.x == 0) g_pf_stamps[blockIdx.x * 4 + (i)] = dev::global_timer_ns();  \
  } while (0)
#define PF_STORE(base, on)                                                             \
  do {                                                                                 \
    if (on) {                                                                          \
      pf_[7] = clock64() - pf_start_;                                                  \
      for (int i_ = 0; i_ < 8; ++i_) g_pf_times[blockIdx.x * 32 + (base) + i_] = pf_[i_]; \
    }                                                                                  \
  } while (0)
#else
#define PF_DECL
#define PF_WAIT(slot, call) (call)
#define PF_MARK(name)
#define PF_ADD(slot, since)
#define PF_STORE(base, on)
#define PF_STAMP(i)
#endif

constexpr int kTcRows = 128;       // query rows per tile (TMEM lanes)
constexpr int kTcItemRows = 256;   // two query tiles per work item
constexpr int kTcTokens = 128;     // tokens per KV tile
constexpr int kTcBlocks = kTcTokens / kBlockSize;
constexpr int kTcThreads = 384;    // 8 softmax warps, producer warp, MMA warp, 2 idle
// registers per thread after the split: launched with 65536 / 384 = 168 each,
// the producer warpgroup gives back to 56 and the softmax warpgroups take
// 224: (224 + 224 + 56) x 128 = 64512 = 168 x 384
constexpr int kTcRegsSoftmax = 224, kTcRegsProducer = 56;
constexpr uint32_t kTcCols = 512;  // TMEM columns: S_0, S_1, O_0, O_1
constexpr float kTcRescale = 8.f;  // log2 of the growth that forces an O rescale

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Tensor-copy store of one box from shared memory (x: element column, a
// multiple of 8 here; y: head; z: token), completed through bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The shared memory of every committed store has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

struct TcSmem {  // head_dim 128, 16-bit: every chunk is [128 rows][128 bytes]
  static constexpr int kChunk = kTcRows * 128;  // 16 KB
  static constexpr int kQ = 0;                  // [2 tiles][2 chunks (d 0-63, 64-127)]
  static constexpr int kK = 4 * kChunk;         // [2 stages][2 chunks]
  static constexpr int kV = kK + 4 * kChunk;    // [2 stages][2 chunks]
  static constexpr int kBars = kV + 4 * kChunk; // mbarriers, item slots
  // per softmax warp: 32 output rows x 64 elements staged for a store
  static constexpr int kOutWarp = 32 * 128;
  static constexpr int kOut = kBars + 1024;
  static constexpr int kBytes = kOut + 8 * kOutWarp + 1024;  // + alignment slack
};
static_assert(TcSmem::kBytes <= 227 * 1024, "tcgen05 prefill shared memory");

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_o, const Params p) {
  constexpr int D = 128;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  using M = dev::Mma<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcSmem::kBars);
  uint64_t* item_full = bars + 0;   // [2] the producer wrote the slot
  uint64_t* item_empty = bars + 2;  // [2] every role has read it
  uint64_t* q_full = bars + 4;
  uint64_t* q_empty = bars + 5;     // the item's last S MMA finished with Q
  uint64_t* k_full = bars + 6;      // [2]
  uint64_t* k_empty = bars + 8;     // [2]
  uint64_t* v_full = bars + 10;     // [2]
  uint64_t* v_empty = bars + 12;    // [2]
  uint64_t* s_full = bars + 14;     // [2] S_w is in TMEM
  uint64_t* p_full = bars + 16;     // [2] P_w is in TMEM (128 arrivals)
  uint64_t* pv_done = bars + 18;    // [2] O_w += P_w V finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  int* s_item = reinterpret_cast<int*>(bars + 21);  // [2]
  uint64_t* drain = bars + 22;      // every MMA issued has finished (error exit)
  // a split item's partial rows are written (8 warp arrivals), then the
  // merge decision is out (1 arrival); the decision word follows
  uint64_t* part_full = bars + 23;
  uint64_t* merge_go = bars + 24;
  int* s_merge = reinterpret_cast<int*>(bars + 25);
  // [2] an item with one query tile alternates its S between the two S
  // buffers (group 1 has no rows then): S of buffer b is in TMEM
  uint64_t* sb_full = bars + 26;
  const uint32_t sbase = dev::smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  PF_STAMP(0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      dev::mbar_init(&item_full[i], 1);
      dev::mbar_init(&item_empty[i], 9);  // 8 softmax warps + the MMA thread
      dev::mbar_init(&k_full[i], 1);
      dev::mbar_init(&k_empty[i], 1);
      dev::mbar_init(&v_full[i], 1);
      dev::mbar_init(&v_empty[i], 1);
      dev::mbar_init(&s_full[i], 1);
      dev::mbar_init(&p_full[i], kTcRows);
      dev::mbar_init(&pv_done[i], 1);
    }
    dev::mbar_init(q_full, 1);
    dev::mbar_init(q_empty, 1);
    dev::mbar_init(drain, 1);
    dev::mbar_init(part_full, 8);
    dev::mbar_init(merge_go, 1);
    dev::mbar_init(&sb_full[0], 1);
    dev::mbar_init(&sb_full[1], 1);
    dev::mbar_fence_init();
    dev::prefetch_tensormap(&tmap_q);
    if (p.out_tma) dev::prefetch_tensormap(&tmap_o);
    dev::prefetch_tensormap(&tmap_k);
    dev::prefetch_tensormap(&tmap_v);
  }
  if (warp == 9) dev::tmem_alloc(tmem_slot, kTcCols);
  dev::tc_fence_before_sync();
  __syncthreads();
  dev::tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();

  const unsigned long long tmo = p.timeout_ns;
  const int G = p.group, Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const bool planned = *reinterpret_cast<volatile int*>(&p.header[kHdrSignature]) == p.signature;
  if (!planned && blockIdx.x == 0 && threadIdx.x == 0) dev::flag_status(p.status, kStatusPlan);
  const int total = planned ? *reinterpret_cast<volatile int*>(&p.header[kHdrTotal]) : 0;
  const bool shared = p.shared_ctx > 0 || p.shared_blocks;
  bool ok = true;
  PF_STAMP(1);

  // what every role decodes from a claimed item
  struct Item {
    int b, qt, first, nblk, ctx, q_first, qlen, g, ntiles, s, ns, slot, grp;
    bool two;  // the second query tile holds valid rows
  };
  auto decode = [&](int x) {
    Item it;
    const int4 u0 = p.units[2 * (x / Hkv)], u1 = p.units[2 * (x / Hkv) + 1];
    it.g = x % Hkv;
    it.b = u0.x;
    it.qt = u0.y;
    it.first = u0.z;  // the item's KV range: blocks first .. first + nblk - 1
    it.nblk = u0.w;
    it.s = u1.x >> 16;  // split index and count
    it.ns = u1.x & 0xffff;
    it.slot = u1.y;     // first partial slot (kRows rows each) and arrival group
    it.grp = u1.z;
    it.ctx = u1.w;
    // shared-prefix mode: the batch's queries are the rows of one sequence
    // (grouped: the group's rows)
    const bool starts = !shared || p.shared_blocks;
    it.q_first = starts ? p.query_start[it.b] : 0;
    it.qlen = starts ? p.query_start[it.b + 1] - it.q_first : p.total_q;
    it.ntiles = (it.nblk + kTcBlocks - 1) / kTcBlocks;
    it.two = it.qt * kTcItemRows + kTcRows < it.qlen * G;
    return it;
  };

  if (warp >= 8) dev::setmaxnreg_dec<kTcRegsProducer>();
  if (warp == 8) {
    // ====================================================== producer warp
    // K/V tiles are loaded evict-first in L2 (evict-last cut DRAM reads from
    // 1.43 to 1.28 times the unique bytes but slowed every measured prefill,
    // most of all the grouped prefix phase)
    const uint64_t policy = dev::l2_policy_evict_first();
    PF_DECL;
    int kt = 0;  // K / V tiles loaded so far
    int qn = 0;  // query-tile loads so far
    for (int n = 0;; ++n) {
      const int slot = n & 1;
      int x = 0;
      if (lane == 0) {
        if (n >= 2)
          ok = PF_WAIT(0, dev::mbar_wait_bounded(&item_empty[slot], ((n >> 1) - 1) & 1, tmo, p.status));
        x = n == 0 ? int(blockIdx.x) : int(gridDim.x) + atomicAdd(&p.header[kHdrNext], 1);
        if (!ok) x = total;  // stop every role
        s_item[slot] = x;
        dev::mbar_arrive(&item_full[slot]);
      }
      x = __shfl_sync(0xffffffffu, x, 0);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (x >= total) break;
      const Item it = decode(x);
      if (lane == 0) {
        if (n >= 1) ok = PF_WAIT(1, dev::mbar_wait_bounded(q_empty, (n - 1) & 1, tmo, p.status));
        if (ok) {
          const int tiles = it.two ? 2 : 1;
          ++qn;
          dev::mbar_arrive_expect_tx(q_full, uint32_t(tiles) * 2 * TcSmem::kChunk);
          for (int w = 0; w < tiles; ++w)
            for (int h = 0; h < 2; ++h) {
              const int zc = it.q_first + it.qt * (kTcItemRows / G) + w * (kTcRows / G);
              asm volatile(
                  "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                  " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sbase + TcSmem::kQ +
                                                           (2 * w + h) * TcSmem::kChunk),
                  "l"(reinterpret_cast<uint64_t>(&tmap_q)), "r"(h * 64), "r"(it.g * G), "r"(zc),
                  "r"(dev::smem_u32(q_full))
                  : "memory");
            }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // table entries, 32 at a time, one per lane
      int tbl = 0, tbl_base = -32;
      for (int j = 0; j < it.ntiles && ok; ++j, ++kt) {
        const int st = kt & 1;
        const int nb = min(kTcBlocks, it.nblk - j * kTcBlocks);
        if ((j * kTcBlocks & ~31) != tbl_base) {
          tbl_base = j * kTcBlocks & ~31;
          tbl = tbl_base + lane < it.nblk
                    ? p.block_tables[size_t(shared ? it.q_first : it.b) * p.max_blocks + it.first +
                                 tbl_base + lane]
                    : 0;
          if (tbl < 0 || tbl >= p.num_blocks) {
            dev::flag_status(p.status, kStatusBounds);
            tbl = 0;
          }
        }
        const int phys = __shfl_sync(0xffffffffu, tbl, (j * kTcBlocks + lane) & 31);
        for (int kind = 0; kind < 2 && ok; ++kind) {  // K, then V
          uint64_t* full = kind == 0 ? &k_full[st] : &v_full[st];
          uint64_t* empty = kind == 0 ? &k_empty[st] : &v_empty[st];
          if (lane == 0) {
            if (kt >= 2)
              ok = PF_WAIT(2 + kind, dev::mbar_wait_bounded(empty, ((kt >> 1) - 1) & 1, tmo, p.status));
            if (ok) dev::mbar_arrive_expect_tx(full, uint32_t(nb) * 4 * 1024);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          // lane jb < nb copies block jb of the tile (both 64-column halves)
          if (lane < nb) {
            const int y = (phys * Hkv + it.g) * kBlockSize;
            uint8_t* dst = smem + (kind == 0 ? TcSmem::kK : TcSmem::kV) +
                           st * 2 * TcSmem::kChunk + lane * 2048;
            const CUtensorMap* map = kind == 0 ? &tmap_k : &tmap_v;
            for (int h = 0; h < 2; ++h)
              dev::tma_load_2d(dst + h * TcSmem::kChunk, map, h * 64, y, full, policy);
          }
        }
      }
      if (!ok) break;
    }
    PF_STORE(24, lane == 0);
    if (lane == 0) {
      // copies still in flight land before the CTA leaves
      if (qn > 0) dev::mbar_wait_bounded(q_full, (qn - 1) & 1, tmo, p.status);
      for (int k = max(0, kt - 2); k < kt; ++k) {
        dev::mbar_wait_bounded(&k_full[k & 1], (k >> 1) & 1, tmo, p.status);
        dev::mbar_wait_bounded(&v_full[k & 1], (k >> 1) & 1, tmo, p.status);
      }
    }
  } else if (warp == 9) {
    // ====================================================== MMA warp
    // The whole warp runs the loop (descriptors stay warp-uniform); the lane
    // elected here issues every MMA and commit.
    const uint32_t leader = dev::elect_one();
    const uint32_t idesc_s = dev::mma_idesc_f16(kBf16, kTcRows, kTcTokens, false);
    const uint32_t idesc_o = dev::mma_idesc_f16(kBf16, kTcRows, D, true);
    // operand descriptors of the tiles' first bytes; a step adds its byte
    // offset / 16 to the address field (the low 14 bits: below 256 KB of
    // shared memory an offset never carries out of it)
    const uint64_t desc_q = dev::smem_desc_sw128(sbase + TcSmem::kQ, 16, 1024);
    const uint64_t desc_k = dev::smem_desc_sw128(sbase + TcSmem::kK, 16, 1024);
    const uint64_t desc_v = dev::smem_desc_sw128(sbase + TcSmem::kV, TcSmem::kChunk, 1024);
    // every lane waits; the warp goes on only if every lane saw the phase
    auto wait = [&](uint64_t* bar, int parity) -> bool {
      return __all_sync(0xffffffffu, dev::mbar_wait_bounded(bar, uint32_t(parity), tmo, p.status));
    };
    int kt = 0;          // K / V tiles consumed
    int pv[2] = {0, 0};  // P V products issued per query tile
    PF_DECL;
    for (int n = 0; ok; ++n) {
      const int slot = n & 1;
      if (!PF_WAIT(0, wait(&item_full[slot], (n >> 1) & 1))) {
        ok = false;
        break;
      }
      const int x = *reinterpret_cast<volatile int*>(&s_item[slot]);
      __syncwarp();
      if (leader) dev::mbar_arrive(&item_empty[slot]);
      if (x >= total) break;
      const Item it = decode(x);
      const int tiles = it.two ? 2 : 1;
      ok = PF_WAIT(1, wait(q_full, n & 1));
      // S_w = Q_w K_j^T once O_w += P_w V of the previous tile has finished
      // (P_w sits in S_w's columns)
      auto issue_s = [&](int w, int st) -> bool {
        if (pv[w] > 0 && !PF_WAIT(5, wait(&pv_done[w], (pv[w] - 1) & 1))) return false;
        dev::tc_fence_after_sync();
        const uint64_t a = desc_q + uint64_t((w * 2 * TcSmem::kChunk) >> 4);
        const uint64_t bk = desc_k + uint64_t((st * 2 * TcSmem::kChunk) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = uint64_t(((kk >> 2) * TcSmem::kChunk + (kk & 3) * 32) >> 4);
          dev::tc_mma_ss_leader(tmem + w * 128, a + off, bk + off, idesc_s, uint32_t(kk), leader);
        }
        dev::tc_commit_leader(&s_full[w], leader);
        return true;
      };
      // O_w += P V, P read from S buffer `buf` (w, or the alternating buffer
      // of a one-tile item)
      auto issue_pv = [&](int w, int j, int st, int buf) -> bool {
        if (!PF_WAIT(4, wait(&p_full[w], pv[w] & 1))) return false;
        dev::tc_fence_after_sync();
        const uint64_t bv = desc_v + uint64_t((st * 2 * TcSmem::kChunk) >> 4);
        const uint32_t d = tmem + 256 + w * 128, pa = tmem + buf * 128;
        dev::tc_mma_ts_leader(d, pa, bv, idesc_o, uint32_t(j), leader);
#pragma unroll
        for (int kk = 1; kk < kTcTokens / 16; ++kk)
          dev::tc_mma_ts_leader(d, pa + kk * 8, bv + uint64_t((kk * 2048) >> 4), idesc_o, 1u, leader);
        dev::tc_commit_leader(&pv_done[w], leader);
        ++pv[w];
        return true;
      };
      if (tiles == 2) {
        // prologue: S of the first tile for both query tiles
        if (ok) ok = PF_WAIT(2, wait(&k_full[kt & 1], (kt >> 1) & 1));
        for (int w = 0; w < tiles && ok; ++w) ok = issue_s(w, kt & 1);
        if (ok) {
          dev::tc_commit_leader(&k_empty[kt & 1], leader);
          if (it.ntiles == 1) dev::tc_commit_leader(q_empty, leader);
        }
        for (int j = 0; j < it.ntiles && ok; ++j) {
          const int st = (kt + j) & 1, nst = (kt + j + 1) & 1;
          const bool more = j + 1 < it.ntiles;
          ok = PF_WAIT(3, wait(&v_full[st], ((kt + j) >> 1) & 1));
          if (ok) ok = issue_pv(0, j, st, 0);
          if (ok && more) {
            ok = PF_WAIT(2, wait(&k_full[nst], ((kt + j + 1) >> 1) & 1));
            if (ok) ok = issue_s(0, nst);
          }
          if (ok) ok = issue_pv(1, j, st, 1);
          if (ok) dev::tc_commit_leader(&v_empty[st], leader);
          if (ok && more) ok = issue_s(1, nst);
          if (ok && more) {
            dev::tc_commit_leader(&k_empty[nst], leader);
            if (j + 2 == it.ntiles) dev::tc_commit_leader(q_empty, leader);
          }
        }
      } else {
        // One query tile: S of tile j goes to S buffer j & 1, so the next
        // tile's S runs while the softmax works on this one.  The buffer's
        // last P was read by the P V two tiles back (the item's tile j - 2,
        // or for j < 2 the previous item's P V, all finished once the newest
        // has); that P V is always the newest issued when S waits for it.
        const int pv0 = pv[0];
        auto issue_s1 = [&](int j, int st) -> bool {
          const int need = j >= 2 ? pv0 + j - 2 : pv0 - 1;
          if (need >= 0 && !PF_WAIT(5, wait(&pv_done[0], need & 1))) return false;
          // buffer 1 last held group 1's P if a two-query-tile item came
          // before: its newest P V came after group 0's
          if (j < 2 && pv[1] > 0 && !PF_WAIT(5, wait(&pv_done[1], (pv[1] - 1) & 1))) return false;
          dev::tc_fence_after_sync();
          const uint64_t bk = desc_k + uint64_t((st * 2 * TcSmem::kChunk) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = uint64_t(((kk >> 2) * TcSmem::kChunk + (kk & 3) * 32) >> 4);
            dev::tc_mma_ss_leader(tmem + (j & 1) * 128, desc_q + off, bk + off, idesc_s,
                                  uint32_t(kk), leader);
          }
          dev::tc_commit_leader(&sb_full[j & 1], leader);
          return true;
        };
        const int pro = it.ntiles < 2 ? it.ntiles : 2;
        for (int j = 0; j < pro && ok; ++j) {
          const int st = (kt + j) & 1;
          ok = PF_WAIT(2, wait(&k_full[st], ((kt + j) >> 1) & 1));
          if (ok) ok = issue_s1(j, st);
          if (ok) dev::tc_commit_leader(&k_empty[st], leader);
        }
        if (ok && it.ntiles <= 2) dev::tc_commit_leader(q_empty, leader);
        for (int j = 0; j < it.ntiles && ok; ++j) {
          const int st = (kt + j) & 1;  // also the stage of tile j + 2
          ok = PF_WAIT(3, wait(&v_full[st], ((kt + j) >> 1) & 1));
          if (ok) ok = issue_pv(0, j, st, j & 1);
          if (ok) dev::tc_commit_leader(&v_empty[st], leader);
          if (ok && j + 2 < it.ntiles) {
            ok = PF_WAIT(2, wait(&k_full[st], ((kt + j + 2) >> 1) & 1));
            if (ok) ok = issue_s1(j + 2, st);
            if (ok) {
              dev::tc_commit_leader(&k_empty[st], leader);
              if (j + 3 == it.ntiles) dev::tc_commit_leader(q_empty, leader);
            }
          }
        }
      }
      kt += it.ntiles;
    }
    PF_STORE(0, leader != 0);
    if (!ok) {
      // a wait ran out: let the MMAs in flight finish before TMEM is freed
      dev::tc_commit_leader(drain, leader);
      dev::mbar_wait_bounded(drain, 0, tmo, p.status);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ====================================================== softmax warps
    dev::setmaxnreg_inc<kTcRegsSoftmax>();
    const int w = warp >> 2;              // query tile of this group
    const int r = threadIdx.x & 127;      // row of the tile = TMEM lane
    const uint32_t lanes = uint32_t((warp & 3) * 32) << 16;
    const uint32_t t_o = tmem + lanes + 256 + w * 128;
    const float sl2 = p.scale_log2;       // > 0 on this path
    int cnt = 0;                          // tiles of this group so far
    int sfw = 0;                          // waits on s_full[w] (two-tile items)
    int sbw[2] = {0, 0};                  // waits on sb_full[b] (one-tile items, group 0)
    int merges = 0;                       // split items merged in-kernel so far
    int kt = 0;                           // K / V tiles so far (group 0 sees them all)
    PF_DECL;
    for (int n = 0;; ++n) {
      const int slot = n & 1;
      if (!PF_WAIT(0, dev::mbar_wait_bounded(&item_full[slot], (n >> 1) & 1, tmo, p.status))) {
        ok = false;
        break;
      }
      const int x = *reinterpret_cast<volatile int*>(&s_item[slot]);
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&item_empty[slot]);
      if (x >= total) break;
      const Item it = decode(x);
      // a split item's rows are merged here unless the caller merges them
      const bool merge_here = it.ns > 1 && !p.defer_merge;
      if (w == 1 && !it.two) {
        // no rows here; still pass this item's merge phase with group 0, so
        // that no later wait can take an old phase for its own
        if (merge_here) {
          if (!dev::mbar_wait_bounded(merge_go, merges & 1, tmo, p.status)) {
            ok = false;
            break;
          }
          ++merges;
        }
        continue;
      }
      const int gr = it.qt * kTcItemRows + w * kTcRows + r;
      const bool valid = gr < it.qlen * G;
      // tokens past the context or past the item's blocks (a split's last
      // tile) are never read into the result
      const int bound = min(it.ctx, (it.first + it.nblk) * kBlockSize);
      // the row's last visible token: causal within the chunk; in
      // shared-prefix mode every row sees the (item's part of the) prefix
      const int pos = valid ? min(shared ? it.ctx - 1 : it.ctx - it.qlen + gr / G, bound - 1) : -1;
      float mref = -INFINITY, l = 0.f;
      for (int j = 0; j < it.ntiles && ok; ++j, ++cnt) {
        // this tile's S buffer: the group's own, or (one query tile) the
        // buffer the tiles alternate over
        const int buf = it.two ? w : (j & 1);
        uint64_t* sbar = it.two ? &s_full[w] : &sb_full[buf];
        const int spar = it.two ? (sfw++ & 1) : (sbw[buf]++ & 1);
        if (!PF_WAIT(1, dev::mbar_wait_bounded(sbar, uint32_t(spar), tmo, p.status))) {
          ok = false;
          break;
        }
        PF_MARK(pf_tile);
        dev::tc_fence_after_sync();
        const uint32_t t_s = tmem + lanes + buf * 128;
        const int t0 = it.first * kBlockSize + j * kTcTokens;  // first token of the tile
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) dev::tmem_ld32(t_s + 32 * c, sv[c]);
        dev::tmem_wait_ld();
        PF_ADD(5, pf_tile);
        PF_MARK(pf_math);
        if (t0 + kTcTokens - 1 > pos) {
          // columns past the row's position (causal, context) do not count
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (t0 + 32 * c + i > pos) sv[c][i] = __float_as_uint(-INFINITY);
        }
        // One query tile: this tile's S did not wait for the previous P V.
        // Wait for it before touching O_w or announcing P, so that at most
        // one P V of this group is ever outstanding: the parity waits on
        // pv_done (here and in the epilogue) and the MMA warp's wait on
        // p_full then never see a barrier two phases ahead.
        bool pv_waited = it.two || j == 0;
        auto wait_prev_pv = [&]() -> bool {
          if (pv_waited) return true;
          pv_waited = true;
          if (!PF_WAIT(3, dev::mbar_wait_bounded(&pv_done[w], (cnt - 1) & 1, tmo, p.status)))
            return false;
          dev::tc_fence_after_sync();
          return true;
        };
        // row maximum: eight independent chains of three-input maxima
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t* v = &sv[k >> 1][16 * (k & 1)];
          float m = dev::fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
          for (int i = 3; i < 15; i += 2) m = dev::fmax3(m, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
          m8[k] = fmaxf(m, __uint_as_float(v[15]));
        }
        float mx = dev::fmax3(dev::fmax3(m8[0], m8[1], m8[2]), dev::fmax3(m8[3], m8[4], m8[5]),
                              fmaxf(m8[6], m8[7])) * sl2;
        if (mx > mref + kTcRescale) {  // also the row's first unmasked column
          if (mref != -INFINITY) {
            // O_w holds every earlier tile once the previous P V has finished
            // (with two query tiles S_w was issued only after it; one tile's
            // S runs ahead, so wait for it): rescale it in TMEM
            if (!wait_prev_pv()) {
              ok = false;
              break;
            }
            const float a = dev::fast_exp2(mref - mx);
            l *= a;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t ov[32];
              dev::tmem_ld32(t_o + 32 * c, ov);
              dev::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * a);
              dev::tmem_st32(t_o + 32 * c, ov);
            }
          }
          mref = mx;
        }
        // P = 2^(s scale log2 e - ref) in the input type, over S's first 64
        // columns; masked columns (-inf) give 0.  A row with nothing visible
        // yet (ref -inf) uses 0 as its reference: every p is 0 then.
        const float nref = mref == -INFINITY ? 0.f : -mref;
        float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            dev::fma2_scalar(x0, x1, __uint_as_float(sv[c][2 * i]), __uint_as_float(sv[c][2 * i + 1]),
                             sl2, nref);
            const float e0 = dev::fast_exp2(x0), e1 = dev::fast_exp2(x1);
            dev::add2(acc[i & 3][0], acc[i & 3][1], e0, e1);
            sv[c >> 1][16 * (c & 1) + i] = M::pack(e0, e1);
          }
        }
        l += ((acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1])) +
             ((acc[2][0] + acc[2][1]) + (acc[3][0] + acc[3][1]));
        PF_ADD(6, pf_math);
        if (!wait_prev_pv()) {
          ok = false;
          break;
        }
        dev::tmem_st32(t_s, sv[0]);
        dev::tmem_st32(t_s + 32, sv[1]);
        if (w == 0 && t0 + kTcTokens > bound) {
          // rows of the last V tile past the context or past the loaded
          // blocks are zeroed, so whatever bits they hold meet only p = 0
          if (!dev::mbar_wait_bounded(&v_full[kt & 1], (kt >> 1) & 1, tmo, p.status)) ok = false;
          if (ok && t0 + r >= bound) {
            // (each row's 16-byte chunks in an order rotated by the row, so
            // the warp's 32 rows, 128 bytes apart, do not all hit one bank)
            uint8_t* vrow = smem + TcSmem::kV + (kt & 1) * 2 * TcSmem::kChunk + r * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int q16 = 0; q16 < 8; ++q16)
                *reinterpret_cast<uint4*>(vrow + h * TcSmem::kChunk + ((q16 + r) & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
          }
          dev::fence_proxy_async_smem();
        }
        if (w == 0) ++kt;
        dev::tmem_wait_st();
        dev::tc_fence_before_sync();
        dev::mbar_arrive(&p_full[w]);
        PF_ADD(2, pf_tile);
      }
      if (!ok) break;
      // O_w is complete once the last P V has finished: normalise and write
      if (!PF_WAIT(3, dev::mbar_wait_bounded(&pv_done[w], (cnt - 1) & 1, tmo, p.status))) {
        ok = false;
        break;
      }
      PF_MARK(pf_epi);
      dev::tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t ov[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) dev::tmem_ld32(t_o + 32 * c, ov[c]);
      dev::tmem_wait_ld();
      if (merge_here) {
        // ---- one of ns splits of this (query block, KV head): its rows'
        // normalised o and base-2 log-sum-exp go to the workspace; the CTA
        // that completes the set merges every row of it.  Slots are counted
        // in kRows-row units: this item's split s starts at row
        // ((slot / (256 / kRows) + s) * Hkv + g) * 256.
        const size_t pstride = size_t(Hkv) * kTcItemRows;
        const size_t pbase =
            (size_t(it.slot / (kTcItemRows / kRows)) * Hkv + it.g) * kTcItemRows + w * kTcRows + r;
        if (valid) {  // rows past the chunk have no partial results (nor a merge)
          float* prow = p.part_o + (pbase + it.s * pstride) * D;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __float_as_uint(__uint_as_float(ov[c][8 * i + e]) * inv);
              dev::st_global_v8(prow + 32 * c + 8 * i, f);
            }
          p.part_lse[pbase + it.s * pstride] = l > 0.f ? mref + log2f(l) : -INFINITY;
        }
        // every participating warp's rows are written (a lone first tile
        // arrives for the absent second one too); one thread counts the split
        __syncwarp();
        if (lane == 0) dev::mbar_arrive_count(part_full, it.two ? 1 : 2);
        if (threadIdx.x == 0) {
          int decision = -1;  // -1: a wait ran out
          if (dev::mbar_wait_bounded(part_full, merges & 1, tmo, p.status))
            decision = dev::atom_add_acq_rel_gpu(&p.arrivals[size_t(it.grp) * Hkv + it.g], 1) ==
                               it.ns - 1
                           ? 1
                           : 0;
          *reinterpret_cast<volatile int*>(s_merge) = decision;
          dev::mbar_arrive(merge_go);
        }
        if (!dev::mbar_wait_bounded(merge_go, merges & 1, tmo, p.status)) ok = false;
        ++merges;
        const int decision = ok ? *reinterpret_cast<volatile int*>(s_merge) : -1;
        if (decision < 0) {
          ok = false;
          break;
        }
        if (decision == 1 && valid) {
          // the last split: merge this thread's row over the ns splits
          float mx = -INFINITY;
          for (int sp = 0; sp < it.ns; ++sp)
            mx = fmaxf(mx, __ldcg(&p.part_lse[pbase + sp * pstride]));
          float sum = 0.f;
          for (int sp = 0; sp < it.ns; ++sp) {
            const float x = __ldcg(&p.part_lse[pbase + sp * pstride]);
            sum += x == -INFINITY ? 0.f : dev::fast_exp2(x - mx);
          }
          const float rs = sum > 0.f ? 1.f / sum : 0.f;
          T* orow = static_cast<T*>(p.out) + (size_t(it.q_first + gr / G) * Hq + it.g * G + gr % G) * D;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {  // 32 columns at a time
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = 0.f;
            for (int sp = 0; sp < it.ns; ++sp) {
              const float x = __ldcg(&p.part_lse[pbase + sp * pstride]);
              const float wgt = x == -INFINITY ? 0.f : dev::fast_exp2(x - mx) * rs;
              const float4* src =
                  reinterpret_cast<const float4*>(p.part_o + (pbase + sp * pstride) * D + 32 * c);
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const float4 v = __ldcg(src + q4);
                acc[4 * q4] += wgt * v.x;
                acc[4 * q4 + 1] += wgt * v.y;
                acc[4 * q4 + 2] += wgt * v.z;
                acc[4 * q4 + 3] += wgt * v.w;
              }
            }
            {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(orow + 32 * c + 8 * i) =
                    make_uint4(M::pack(acc[8 * i], acc[8 * i + 1]), M::pack(acc[8 * i + 2], acc[8 * i + 3]),
                               M::pack(acc[8 * i + 4], acc[8 * i + 5]),
                               M::pack(acc[8 * i + 6], acc[8 * i + 7]));
            }
          }
        }
        // ready for the next run on this plan
        if (decision == 1 && threadIdx.x == 0) p.arrivals[size_t(it.grp) * Hkv + it.g] = 0;
      } else if (valid && shared) {
        // fp32 o (normalised) and the base-2 log-sum-exp of the row
        const size_t hrow = size_t(it.q_first + gr / G) * Hq + it.g * G + gr % G;
        const size_t rows = size_t(p.total_q) * Hq;  // split s writes part s
        float* crow = p.cas_o + (size_t(it.s) * rows + hrow) * D;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __float_as_uint(__uint_as_float(ov[c][8 * i + e]) * inv);
            dev::st_global_v8(crow + 32 * c + 8 * i, f);
          }
        p.cas_lse[size_t(it.s) * rows + hrow] = l > 0.f ? mref + log2f(l) : -INFINITY;
      } else if (p.out_tma && __all_sync(0xffffffffu, valid)) {
        // The warp's 32 rows are 32 / G tokens x the G heads of the group:
        // one box of the output's tensor map per 64 columns.  Each row goes
        // to shared memory in the box's 128-byte-swizzled layout (so the 32
        // rows' 16-byte stores spread over every bank), then one lane stores
        // the box; the staging buffer is reused once the previous store has
        // read it.
        const uint32_t stage = sbase + TcSmem::kOut + warp * TcSmem::kOutWarp;
        const int tok0 = it.q_first + (gr - lane) / G;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t* x = &ov[2 * h + (k >> 2)][8 * (k & 3)];
            st_shared_v4(stage + lane * 128 + ((k ^ (lane & 7)) << 4),
                         M::pack(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                         M::pack(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                         M::pack(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                         M::pack(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
          }
          dev::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmap_o, stage, h * 64, it.g * G, tok0);
            bulk_commit_group();
          }
        }
      } else if (valid) {
        T* orow = static_cast<T*>(p.out) +
                  (size_t(it.q_first + gr / G) * Hq + it.g * G + gr % G) * D;
        // a row is 256 bytes: whole 32-byte sectors per store when the
        // output is 32-byte aligned, 16-byte stores otherwise
        const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = M::pack(__uint_as_float(ov[c][2 * i]) * inv, __uint_as_float(ov[c][2 * i + 1]) * inv);
          if (wide) {
            dev::st_global_v8(orow + 32 * c, pk);
            dev::st_global_v8(orow + 32 * c + 16, pk + 8);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(orow + 32 * c + 8 * i) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      // O_w is read: the next item's first P V may overwrite it
      dev::tc_fence_before_sync();
      PF_ADD(4, pf_epi);
    }
    if (p.out_tma && lane == 0) bulk_wait_all();  // the output stores have landed
    PF_STORE(8 + 8 * w, r == 0);
  }
  PF_STAMP(2);
  dev::tc_fence_before_sync();
  const bool all_ok = __syncthreads_and(ok);
  if (warp == 9) {
    dev::tc_fence_after_sync();
    dev::tmem_dealloc(tmem, kTcCols);
  }
  PF_STAMP(3);
  if (threadIdx.x == 0 && planned && all_ok) {
    __threadfence();
    if (atomicAdd(&p.header[kHdrDone], 1) == int(gridDim.x) - 1) {
      atomicExch(&p.header[kHdrNext], 0);
      atomicExch(&p.header[kHdrDone], 0);
    }
  }
}

// --------------------------------------------------------------- fp32 path
// One warp per (query row, query head): a decode over the row's causal prefix.
template <int D>
__global__ void __launch_bounds__(128) prefill_f32_kernel(const Params p) {
  constexpr int E = D / 32;
  const long long unit = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (unit >= (long long)p.total_q * p.num_q_heads) return;
  const int row = int(unit / p.num_q_heads), h = int(unit % p.num_q_heads);
  // the sequence of this row: query_start is sorted, binary search
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.query_start[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  if (row < p.query_start[b] || row >= p.query_start[b + 1]) return;  // no sequence's row
  const int qlen = p.query_start[b + 1] - p.query_start[b];
  const int ctx = p.context_lens[b];
  const int cap = p.max_blocks * kBlockSize;
  if (ctx < 0 || ctx > cap || qlen > ctx) {
    if (lane == 0) dev::flag_status(p.status, kStatusBounds);
    return;
  }
  const int pos = ctx - qlen + (row - p.query_start[b]);
  const int g = h / p.group;
  const float* qv = static_cast<const float*>(p.q) + (size_t(row) * p.num_q_heads + h) * D + lane * E;
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
  for (int t = 0; t <= pos; ++t) {
    int phys = table[t / kBlockSize];
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) dev::flag_status(p.status, kStatusBounds);
      phys = 0;
    }
    const size_t r = ((size_t(phys) * p.num_kv_heads + g) * kBlockSize + t % kBlockSize) * D + lane * E;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(qr[e], k_cache[r + e], dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float sc = dot * p.scale;
    const float mn = fmaxf(m, sc);
    const float a = expf(m - mn), pw = expf(sc - mn);
    l = l * a + pw;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = acc[e] * a + pw * v_cache[r + e];
    m = mn;
  }
  float* out = static_cast<float*>(p.out) + (size_t(row) * p.num_q_heads + h) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = acc[e] / l;
}

}  // namespace prefill
}  // namespace pa

// ====================================================================== host
namespace pa {
namespace prefill {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int error = 0;
  int sms = 0;
  int ctas_per_sm[2][2] = {{0, 0}, {0, 0}};  // [bf16?][head_dim 128?]
  bool tc_ok = false;                        // tcgen05 kernel configured
};

// The tcgen05 kernel serves 16-bit, head_dim 128 and groups dividing its
// 128-row tile (the mma.sync kernel the rest); PA_PREFILL_TC=0 turns it off
// (read once per process).
bool tc_wanted() {
  static const bool on = [] {
    const char* v = std::getenv("PA_PREFILL_TC");
    return v ? std::atoi(v) != 0 : true;
  }();
  return on;
}
DeviceState g_dev[kMaxDevices];

template <typename T, int D>
cudaError_t configure(int* ctas_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Smem<D>::kBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, prefill_kernel<T, D>,
                                                       kWarps * 32, Smem<D>::kBytes);
}

int device_setup(int device) {
  DeviceState& st = g_dev[device];
  std::call_once(st.once, [&] {
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      st.error = PA_ERR_CUDA;
      return;
    }
    cudaError_t e = configure<__nv_bfloat16, 128>(&st.ctas_per_sm[1][1]);
    if (e == cudaSuccess) e = configure<__nv_bfloat16, 64>(&st.ctas_per_sm[1][0]);
    if (e == cudaSuccess) e = configure<__half, 128>(&st.ctas_per_sm[0][1]);
    if (e == cudaSuccess) e = configure<__half, 64>(&st.ctas_per_sm[0][0]);
    st.error = e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    for (int a = 0; a < 2; ++a)
      for (int d = 0; d < 2; ++d)
        if (st.error == PA_OK && st.ctas_per_sm[a][d] < 1) st.error = PA_ERR_UNSUPPORTED;
    if (st.error == PA_OK) {
      st.tc_ok = cudaFuncSetAttribute(prefill_tc_kernel<__nv_bfloat16>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      TcSmem::kBytes) == cudaSuccess &&
                 cudaFuncSetAttribute(prefill_tc_kernel<__half>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      TcSmem::kBytes) == cudaSuccess;
      cudaGetLastError();
    }
  });
  if (st.error != PA_OK) return fail(st.error, "prefill: per-device set-up failed on device %d", device);
  return PA_OK;
}

bool prepare(Params& prm, const Layout& lay, int device, int dtype, void* workspace);
int launch_plan(const Params& prm, bool use_tc, cudaStream_t s, const char* who);
int launch_attention(const Params& prm, bool use_tc, int dtype, cudaStream_t s, const char* who);

int check_shapes(int num_seqs, int total_q, int num_q_heads, int num_kv_heads, int head_dim,
                 int max_blocks_per_seq, int dtype, const char* who) {
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "%s: unknown dtype %d", who, dtype);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d (64 or 128)", who, head_dim);
  if (num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: sizes must be positive", who);
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "%s: num_q_heads %% num_kv_heads != 0", who);
  if (num_q_heads / num_kv_heads > kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "%s: %d query heads per KV head (max %d)", who,
                num_q_heads / num_kv_heads, kMaxGroup);
  if (double(max_blocks_per_seq) * kBlockSize >= 2147483647.0 ||
      double(total_q) * num_q_heads >= 2147483647.0)
    return fail(PA_ERR_INVALID_ARG, "%s: sizes too large", who);
  return PA_OK;
}

}  // namespace
}  // namespace prefill
}  // namespace pa

using namespace pa;
using namespace pa::prefill;

extern "C" {

#ifdef PA_PROFILE_TIMES
PA_API int pa_profile_prefill_stamps(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, pa::prefill::g_pf_stamps, size_t(n) * sizeof(unsigned long long)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}
PA_API int pa_profile_prefill_times(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, pa::prefill::g_pf_times, size_t(n) * sizeof(unsigned long long)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}
#endif


PA_API int pa_paged_attention_prefill_workspace_size(int num_seqs, int total_q, int num_q_heads,
                                                     int num_kv_heads, int head_dim,
                                                     size_t* bytes) {
  if (!bytes) return fail(PA_ERR_INVALID_ARG, "prefill_workspace_size: bytes is NULL");
  if (num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "prefill_workspace_size: bad sizes");
  *bytes = workspace_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim).total;
  return PA_OK;
}

}  // extern "C"

namespace pa {
namespace prefill {
namespace {

enum class Mode { kPlanAndRun, kPlanOnly, kRunOnly };

// Validation, then the plan and / or the attention kernel.  The plan reads
// only context_lens and query_start (and the sizes); q, the caches, the
// tables and out may be NULL for Mode::kPlanOnly.
int prefill_entry(Mode mode, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens,
                  const int32_t* query_start, int num_seqs, int total_q, int num_q_heads,
                  int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                  float scale, int dtype, void* out, void* workspace, size_t workspace_bytes,
                  void* stream, const char* who) {
  int rc = check_shapes(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim,
                        max_blocks_per_seq, dtype, who);
  if (rc != PA_OK) return rc;
  if (num_seqs == 0 || total_q == 0) return PA_OK;
  const bool runs = mode != Mode::kPlanOnly;
  if (!context_lens || !query_start)
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (runs && (!q || !k_cache || !v_cache || !block_tables || !out))
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  auto misaligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) != 0; };
  if (runs && (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out)))
    return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", who);
  if (runs && (num_blocks <= 0 || double(num_blocks) * num_kv_heads * kBlockSize >= 2147483647.0))
    return fail(PA_ERR_INVALID_ARG, "%s: bad num_blocks", who);
  const Layout lay = workspace_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace must be non-NULL and 256-byte aligned", who);
  if (workspace_bytes < lay.total)
    return fail(PA_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                lay.total);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "%s: no current CUDA device", who);
  rc = device_setup(device);
  if (rc != PA_OK) return rc;
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  Params prm = {};
  prm.q = q;
  prm.k_cache = k_cache;
  prm.v_cache = v_cache;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.query_start = query_start;
  prm.num_seqs = num_seqs;
  prm.total_q = total_q;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = num_q_heads / num_kv_heads;
  prm.head_dim = head_dim;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = num_blocks;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.status = status;
  prm.timeout_ns = 1000000000ull;

  if (dtype == PA_F32) {
    // one warp per (row, head) needs no plan
    if (!runs) return PA_OK;
    const long long units = (long long)total_q * num_q_heads;
    const int blocks = int((units + 3) / 4);
    if (head_dim == 64)
      prefill_f32_kernel<64><<<blocks, 128, 0, s>>>(prm);
    else
      prefill_f32_kernel<128><<<blocks, 128, 0, s>>>(prm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s (fp32): launch failed: %s", who, cudaGetErrorString(e));
    return PA_OK;
  }
  const bool use_tc = prepare(prm, lay, device, dtype, workspace);
  if (mode != Mode::kRunOnly) {
    rc = launch_plan(prm, use_tc, s, who);
    if (rc != PA_OK) return rc;
  }
  return runs ? launch_attention(prm, use_tc, dtype, s, who) : PA_OK;
}

}  // namespace
}  // namespace prefill
}  // namespace pa

extern "C" {

PA_API int pa_paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      const int32_t* query_start, int num_seqs, int total_q,
                                      int num_q_heads, int num_kv_heads, int head_dim,
                                      int max_blocks_per_seq, int num_blocks, float scale,
                                      int dtype, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_prefill");
  return pa::prefill::prefill_entry(pa::prefill::Mode::kPlanAndRun, q, k_cache, v_cache,
                                    block_tables, context_lens, query_start, num_seqs, total_q,
                                    num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                    num_blocks, scale, dtype, out, workspace, workspace_bytes,
                                    stream, "paged_attention_prefill");
}

PA_API int pa_paged_attention_prefill_plan(const int32_t* context_lens,
                                           const int32_t* query_start, int num_seqs,
                                           int total_q, int num_q_heads, int num_kv_heads,
                                           int head_dim, int max_blocks_per_seq, float scale,
                                           int dtype, void* workspace, size_t workspace_bytes,
                                           void* stream) {
  PA_TRACE("pa_paged_attention_prefill_plan");
  return pa::prefill::prefill_entry(pa::prefill::Mode::kPlanOnly, nullptr, nullptr, nullptr,
                                    nullptr, context_lens, query_start, num_seqs, total_q,
                                    num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, 0,
                                    scale, dtype, nullptr, workspace, workspace_bytes, stream,
                                    "paged_attention_prefill_plan");
}

PA_API int pa_paged_attention_prefill_run(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, const int32_t* context_lens,
                                          const int32_t* query_start, int num_seqs, int total_q,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq, int num_blocks, float scale,
                                          int dtype, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  PA_TRACE("pa_paged_attention_prefill_run");
  return pa::prefill::prefill_entry(pa::prefill::Mode::kRunOnly, q, k_cache, v_cache,
                                    block_tables, context_lens, query_start, num_seqs, total_q,
                                    num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                    num_blocks, scale, dtype, out, workspace, workspace_bytes,
                                    stream, "paged_attention_prefill_run");
}

}  // extern "C"

namespace pa {
namespace prefill {
namespace {

// The plan-dependent fields of a filled-in Params (16-bit dtypes): which
// kernel runs (its query-block size fixes the plan), the plan's signature and
// the workspace's pieces.  Returns whether the tensor-core kernel runs.
bool prepare(Params& prm, const Layout& lay, int device, int dtype, void* workspace) {
  const DeviceState& st = g_dev[device];
  const bool bf16 = dtype == PA_BF16;
  const int per_sm = st.ctas_per_sm[bf16][prm.head_dim == 128];
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int G = prm.num_q_heads / prm.num_kv_heads;
  const bool use_tc = tc_wanted() && st.tc_ok && prm.head_dim == 128 && prm.scale_log2 > 0.f &&
                      (G == 1 || G == 2 || G == 4 || G == 8);
  prm.ncta = use_tc ? st.sms : st.sms * per_sm;
  // the tcgen05 kernel merges its splits itself, except in the shared-prefix
  // phase, whose parts the cascade combine merges
  prm.defer_merge = use_tc && (prm.shared_ctx > 0 || prm.shared_blocks) ? 1 : 0;
  prm.no_split = 0;
  prm.units_cap = lay.units_cap;
  prm.partial_cap = lay.partial_cap;
  prm.signature = signature_of(prm.num_seqs, prm.total_q, prm.num_q_heads, prm.num_kv_heads,
                               prm.head_dim, prm.max_blocks) ^
                  (prm.shared_ctx << 1) ^ (use_tc ? 0x2A000000 : 0) ^
                  (prm.shared_blocks ? 0x15000000 : 0);
  prm.header = reinterpret_cast<int*>(ws + lay.header);
  prm.units = reinterpret_cast<int4*>(ws + lay.units);
  prm.arrivals = reinterpret_cast<int*>(ws + lay.arrivals);
  prm.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  prm.part_o = reinterpret_cast<float*>(ws + lay.part_o);
  return use_tc;
}

cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// The one-CTA plan kernel: the work list into the workspace.
int launch_plan(const Params& prm, bool use_tc, cudaStream_t s, const char* who) {
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cudaLaunchConfig_t pc = {};
  pc.gridDim = dim3(1);
  pc.blockDim = dim3(kPlanThreads);
  pc.stream = s;
  pc.attrs = attr;
  pc.numAttrs = 1;
  cudaError_t e = use_tc ? cudaLaunchKernelEx(&pc, prefill_plan_kernel<kTcItemRows>, prm)
                         : cudaLaunchKernelEx(&pc, prefill_plan_kernel<kRows>, prm);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: plan launch failed: %s", who, cudaGetErrorString(e));
  return PA_OK;
}

// The attention kernel over a planned workspace.
int launch_attention(const Params& prm_in, bool use_tc, int dtype, cudaStream_t s, const char* who) {
  const bool bf16 = dtype == PA_BF16;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  alignas(64) CUtensorMap mq, mk, mv, mo;
  Params prm = prm_in;
  int rc = cache_tensor_map(&mk, prm.k_cache, bf16, prm.num_blocks, prm.num_kv_heads, prm.head_dim);
  if (rc == PA_OK)
    rc = cache_tensor_map(&mv, prm.v_cache, bf16, prm.num_blocks, prm.num_kv_heads, prm.head_dim);
  if (rc != PA_OK) return rc;
  cudaError_t e;
  if (use_tc) {
    rc = query_tensor_map(&mq, prm.q, bf16, prm.total_q, prm.num_q_heads, prm.head_dim,
                          prm.num_q_heads / prm.num_kv_heads, kTcRows);
    if (rc != PA_OK) return rc;
    // rows to out by tensor-copy stores: a warp's 32 rows at a time (the
    // shared-prefix modes write fp32 parts instead)
    std::memset(&mo, 0, sizeof(mo));
    prm.out_tma = prm.out && prm.shared_ctx == 0 && !prm.shared_blocks &&
                  (reinterpret_cast<uintptr_t>(prm.out) & 15) == 0;
    if (prm.out_tma) {
      rc = output_tensor_map(&mo, prm.out, bf16, prm.total_q, prm.num_q_heads, prm.head_dim,
                             prm.num_q_heads / prm.num_kv_heads, 32);
      if (rc != PA_OK) return rc;
    }
    cudaLaunchConfig_t tc = {};
    tc.gridDim = dim3(prm.ncta);
    tc.blockDim = dim3(kTcThreads);
    tc.dynamicSmemBytes = TcSmem::kBytes;
    tc.stream = s;
    tc.attrs = attr;
    tc.numAttrs = 1;
    e = bf16 ? cudaLaunchKernelEx(&tc, prefill_tc_kernel<__nv_bfloat16>, mq, mk, mv, mo, prm)
             : cudaLaunchKernelEx(&tc, prefill_tc_kernel<__half>, mq, mk, mv, mo, prm);
  } else {
    cudaLaunchConfig_t kc = {};
    kc.gridDim = dim3(prm.ncta);
    kc.blockDim = dim3(kWarps * 32);
    kc.stream = s;
    kc.attrs = attr;
    kc.numAttrs = 1;
    if (prm.head_dim == 128) {
      kc.dynamicSmemBytes = Smem<128>::kBytes;
      e = bf16 ? cudaLaunchKernelEx(&kc, prefill_kernel<__nv_bfloat16, 128>, mk, mv, prm)
               : cudaLaunchKernelEx(&kc, prefill_kernel<__half, 128>, mk, mv, prm);
    } else {
      kc.dynamicSmemBytes = Smem<64>::kBytes;
      e = bf16 ? cudaLaunchKernelEx(&kc, prefill_kernel<__nv_bfloat16, 64>, mk, mv, prm)
               : cudaLaunchKernelEx(&kc, prefill_kernel<__half, 64>, mk, mv, prm);
    }
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace

const int* shared_prefix_split_count(const void* workspace) {
  return static_cast<const int*>(workspace) + kHdrSplits;  // the header is at offset 0
}

const int* shared_prefix_split_blocks(const void* workspace) {
  return static_cast<const int*>(workspace) + kHdrSplitBlocks;
}

size_t shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim) {
  return workspace_layout(num_seqs, num_seqs, num_q_heads, num_kv_heads, head_dim).total;
}

namespace {

// Params of the shared-prefix phase: the batch's decode queries are the rows
// of one sequence over the prefix (no causal mask).
int shared_params(Params& prm, Layout& lay, int& device, const void* q, const void* k_cache,
                  const void* v_cache, const int32_t* block_tables, int prefix_tokens,
                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                  int max_blocks_per_seq, int num_blocks, float scale, float* cas_o,
                  float* cas_lse, size_t workspace_bytes, const char* who) {
  // sized for up to num_seqs groups (one group in the single-prefix mode),
  // so both modes share one layout
  lay = workspace_layout(num_seqs, num_seqs, num_q_heads, num_kv_heads, head_dim);
  if (workspace_bytes < lay.total) return fail(PA_ERR_INVALID_ARG, "%s: workspace too small", who);
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "%s: no current CUDA device", who);
  int rc = device_setup(device);
  if (rc != PA_OK) return rc;
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  prm = Params{};
  prm.q = q;
  prm.k_cache = k_cache;
  prm.v_cache = v_cache;
  prm.block_tables = block_tables;
  prm.num_seqs = 1;
  prm.total_q = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = num_q_heads / num_kv_heads;
  prm.head_dim = head_dim;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = num_blocks;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.status = status;
  prm.timeout_ns = 1000000000ull;
  prm.shared_ctx = prefix_tokens;
  prm.cas_o = cas_o;
  prm.cas_lse = cas_lse;
  return PA_OK;
}

}  // namespace

int shared_prefix_plan(int prefix_tokens, int num_seqs, int num_q_heads, int num_kv_heads,
                       int head_dim, int max_blocks_per_seq, float scale, int dtype,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const char* who = "paged_attention_decode_shared_prefix (prefix plan)";
  Params prm;
  Layout lay;
  int device = 0;
  int rc = shared_params(prm, lay, device, nullptr, nullptr, nullptr, nullptr, prefix_tokens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, 0,
                         scale, nullptr, nullptr, workspace_bytes, who);
  if (rc != PA_OK) return rc;
  const bool use_tc = prepare(prm, lay, device, dtype, workspace);
  return launch_plan(prm, use_tc, stream, who);
}

int shared_prefix_run(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int prefix_tokens, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                      int num_blocks, float scale, int dtype, float* cas_o, float* cas_lse,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const char* who = "paged_attention_decode_shared_prefix (prefix)";
  Params prm;
  Layout lay;
  int device = 0;
  int rc = shared_params(prm, lay, device, q, k_cache, v_cache, block_tables, prefix_tokens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                         num_blocks, scale, cas_o, cas_lse, workspace_bytes, who);
  if (rc != PA_OK) return rc;
  const bool use_tc = prepare(prm, lay, device, dtype, workspace);
  return launch_attention(prm, use_tc, dtype, stream, who);
}

int grouped_prefix_plan(const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_blocks_per_seq, float scale, int dtype, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  const char* who = "paged_attention_decode_grouped_prefix (prefix plan)";
  Params prm;
  Layout lay;
  int device = 0;
  int rc = shared_params(prm, lay, device, nullptr, nullptr, nullptr, nullptr, 0, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, 0, scale,
                         nullptr, nullptr, workspace_bytes, who);
  if (rc != PA_OK) return rc;
  prm.num_seqs = num_groups;
  prm.query_start = group_start;
  prm.shared_blocks = group_blocks;
  const bool use_tc = prepare(prm, lay, device, dtype, workspace);
  return launch_plan(prm, use_tc, stream, who);
}

int grouped_prefix_run(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* group_start,
                       const int32_t* group_blocks, int num_groups, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                       float scale, int dtype, float* cas_o, float* cas_lse, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  const char* who = "paged_attention_decode_grouped_prefix (prefix)";
  Params prm;
  Layout lay;
  int device = 0;
  int rc = shared_params(prm, lay, device, q, k_cache, v_cache, block_tables, 0, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_blocks,
                         scale, cas_o, cas_lse, workspace_bytes, who);
  if (rc != PA_OK) return rc;
  prm.num_seqs = num_groups;
  prm.query_start = group_start;
  prm.shared_blocks = group_blocks;
  const bool use_tc = prepare(prm, lay, device, dtype, workspace);
  return launch_attention(prm, use_tc, dtype, stream, who);
}

int shared_prefix_phase(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int prefix_tokens, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                        int num_blocks, float scale, int dtype, float* cas_o, float* cas_lse,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = shared_prefix_plan(prefix_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                              max_blocks_per_seq, scale, dtype, workspace, workspace_bytes, stream);
  if (rc != PA_OK) return rc;
  return shared_prefix_run(q, k_cache, v_cache, block_tables, prefix_tokens, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_blocks,
                           scale, dtype, cas_o, cas_lse, workspace, workspace_bytes, stream);
}

}  // namespace prefill
}  // namespace pa
