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
//  * persistent attention kernel, one CTA per SM, two warp roles:
//      - scheduler warp: takes work items from a global counter (four at a
//        time, so their dependent global reads overlap), reads each item's
//        block-table entries (range-checked) and bulk-copies the G query rows
//        of (b, g) into a shared-memory item queue;
//      - W math warps: each takes whole items from the queue and streams all
//        their blocks through its own small ring, issuing the 2-D tensor
//        copies (128-byte swizzled, L2 evict-first) of a block's K and V
//        tiles a few blocks before it needs them.  Many independent issuers
//        keep HBM busy; a single issuing thread per CTA could not (each copy
//        instruction costs it hundreds of cycles), and no CTA-wide barrier is
//        needed.  Per 16-token block: S^T = K . Q^T on the tensor cores
//        (m16n8k16, M = the 16 tokens, N = the G <= 8 query heads of the
//        group, K = head_dim), online softmax in base 2 with per-head running
//        max / sum, P rounded to the input type and transposed in registers
//        (movmatrix), O^T += V^T . P^T (M = head_dim rows of V^T via
//        ldmatrix.trans).  Each K/V tile is read from HBM once for the whole
//        query group.  Slots past the context in the last block are zeroed in
//        registers, so whatever bits they hold cannot reach the output.
//    A sequence with one split is written to `out` straight from the
//    warp's registers; otherwise the warp writes (o, lse) to the workspace,
//    publishes it (fence) and counts it (atomic), and the warp that completes
//    the last split of (b, g) merges all splits with log-sum-exp weights (no
//    spinning).  The work and arrival counters return to zero by the end of
//    every run.
//  * Every wait is an mbarrier wait with a time limit; running out sets the
//    timeout bit of the device status word and the warp returns.
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
#include <mutex>
#include <type_traits>

#include "decode.cuh"
#include "device_common.cuh"
#include "pagedattn.h"
#include "status.h"

namespace pa {
namespace decode {

using dev::mbar_arrive;
using dev::mbar_wait_bounded;

// Optional cycle accounting per CTA and warp role, compiled in only with
// -DPA_PROFILE (a separate build used to see where a persistent CTA spends its
// time; the default build has none of it).
#ifdef PA_PROFILE_TIMES
// per (CTA, warp): globaltimer at start of work, at end, blocks consumed
__device__ unsigned long long g_times[2048 * 16 * 3];
#define TIME_MARK(i, v)                                                                     \
  do {                                                                                      \
    if ((threadIdx.x & 31) == 0)                                                            \
      g_times[(blockIdx.x * 16 + (threadIdx.x >> 5)) * 3 + (i)] = (v);                      \
  } while (0)
#else
#define TIME_MARK(i, v)
#endif

#ifdef PA_PROFILE
constexpr int kProfSlots = 16;
__device__ unsigned long long g_prof[2048 * kProfSlots];
#define PROF_T(var) const long long var = clock64()
#define PROF_ADD(slot, t0)                                                                  \
  do {                                                                                      \
    if ((threadIdx.x & 31) == 0)                                                            \
      atomicAdd(&g_prof[blockIdx.x * kProfSlots + (slot)],                                  \
                static_cast<unsigned long long>(clock64() - (t0)));                         \
  } while (0)
#define PROF_INC(slot, v)                                                                   \
  do {                                                                                      \
    if ((threadIdx.x & 31) == 0)                                                            \
      atomicAdd(&g_prof[blockIdx.x * kProfSlots + (slot)], static_cast<unsigned long long>(v)); \
  } while (0)
#else
#define PROF_T(var)
#define PROF_ADD(slot, t0)
#define PROF_INC(slot, v)
#endif

template <int D>
struct alignas(128) ItemSlot {
  int b, g, s, ctx, nblk, nsplit, first, pad0;
  int blocks[kSplitBlocks];
  alignas(16) uint16_t q[kMaxGroup * D];
};

template <int D, int W>
struct Smem {
  static constexpr int kTileBytes = kBlockSize * D * 2;  // one (block, head) tile
  static constexpr int kStageBytes = 2 * kTileBytes;     // K tile + V tile
  static constexpr size_t kItems = size_t(kQueue) * sizeof(ItemSlot<D>);
  // barriers (uint64) + the claim and pushed counters
  static constexpr size_t kBars = size_t(W) * kWarpStages + 2 * kQueue + 1;
  static size_t fixed_bytes(int /*group*/) {
    return 1024 /* alignment slack */ + kItems + kBars * 8 + 16;
  }
  // `stages` is per math warp
  static size_t bytes(int group, int stages) {
    return fixed_bytes(group) + size_t(W) * stages * kStageBytes;
  }
  static int stages_for(int group, size_t budget) {
    const long avail = long(budget) - long(fixed_bytes(group));
    long s = avail / (long(W) * kStageBytes);
    if (s > kWarpStages) s = kWarpStages;
    return int(s);
  }
};

// ------------------------------------------------------------------ plan
// Splits of one sequence are balanced: nsplit = ceil(blocks / 32) splits whose
// sizes differ by at most one block.  Units are then counting-sorted by size,
// largest first, and a sequence's splits stay adjacent in the order.
__device__ __forceinline__ void split_shape(int nblk, int split, int& nsplit, int& base,
                                            int& big) {
  nsplit = (nblk + split - 1) / split;
  base = nsplit ? nblk / nsplit : 0;
  big = nsplit ? nblk - base * nsplit : 0;  // the first `big` splits hold base + 1 blocks
}

__global__ void __launch_bounds__(1024) plan_kernel(const Params p) {
  __shared__ int hist[kSplitBlocks + 2];
  __shared__ int bucket[kSplitBlocks + 2];
  dev::grid_launch_dependents();
  const int tid = threadIdx.x;
  if (tid < kSplitBlocks + 2) hist[tid] = 0;
  __syncthreads();
  const int cap = p.max_blocks * kBlockSize;
  int4* units = reinterpret_cast<int4*>(p.ws.units);

  for (int b = tid; b < p.num_seqs; b += 1024) {
    int ctx = p.context_lens[b];
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
  for (int b = tid; b < p.num_seqs; b += 1024) {
    int ctx = p.context_lens[b];
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    int nsplit, base, big;
    split_shape((ctx + kBlockSize - 1) / kBlockSize, p.split_blocks, nsplit, base, big);
    const int at_big = big ? atomicAdd(&bucket[base + 1], big) : 0;
    const int at_small = nsplit - big ? atomicAdd(&bucket[base], nsplit - big) : 0;
    int first = 0;
    for (int s = 0; s < nsplit; ++s) {
      const int n = s < big ? base + 1 : base;
      const int pos = s < big ? at_big + s : at_small + (s - big);
      units[pos] = make_int4(b, (s << 8) | n, first, ctx);
      first += n;
    }
  }
}

// --------------------------------------------------------- tensor-core path
template <typename T, int D, int W>
__global__ void __launch_bounds__((W + 1) * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  using S = Smem<D, W>;
  using M = dev::Mma<T>;
  constexpr int KT = D / 16;        // 16-wide steps along head_dim
  constexpr int HALVES = D / 64;    // 128-byte TMA boxes per tile row
  constexpr int FIFO = 2;           // items a math warp may hold (1 in work + 1 lookahead)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int G = p.group;
  const int NS = p.stages;  // ring stages per math warp
  uint8_t* rings = smem;
  ItemSlot<D>* items =
      reinterpret_cast<ItemSlot<D>*>(rings + size_t(W) * NS * S::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(items) + S::kItems);
  uint64_t* item_full = full + W * kWarpStages;  // [W][kWarpStages] before it
  uint64_t* item_empty = item_full + kQueue;
  int* claim_ctr = reinterpret_cast<int*>(item_empty + kQueue);
  // items the scheduler has written to the queue so far (only it writes)
  volatile int* pushed = claim_ctr + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef PA_PROFILE_TIMES
  if (threadIdx.x == 0) g_times[(blockIdx.x * 16 + 15) * 3 + 0] = dev::global_timer_ns();
#endif
  if (threadIdx.x == 0) {
    for (int i = 0; i < W * kWarpStages; ++i) dev::mbar_init(&full[i], 1);
    for (int i = 0; i < kQueue; ++i) {
      dev::mbar_init(&item_full[i], 8);  // the lanes of one scheduler group
      dev::mbar_init(&item_empty[i], 1);  // the one math warp that took the item
    }
    *claim_ctr = 0;
    *pushed = 0;
    dev::mbar_fence_init();
  }
  if (warp < W && lane == 0) {
    dev::prefetch_tensormap(&tmap_k);
    dev::prefetch_tensormap(&tmap_v);
  }
  __syncthreads();
  dev::grid_dependency_wait();  // a plan launched just before has completed

  PROF_T(t_kernel);
#ifdef PA_PROFILE_TIMES
  if (threadIdx.x == 0) g_times[(blockIdx.x * 16 + 15) * 3 + 1] = dev::global_timer_ns();
#endif
  const unsigned long long tmo = p.timeout_ns;
  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  const bool planned =
      *reinterpret_cast<volatile int*>(&p.ws.header[kHdrSignature]) == p.signature;

  if (warp == W) {
    // ------------------------------------------------------------ scheduler
    // Four lane groups of 8 fetch four work items at once, so the dependent
    // global round trips of an item (counter -> unit -> table entries) overlap.
    if (!planned) {
      if (lane == 0 && blockIdx.x == 0) dev::flag_status(p.status, kStatusPlan);
    } else {
      // rows of empty sequences are zero
      for (int b = blockIdx.x * 32 + lane; b < p.num_seqs; b += gridDim.x * 32) {
        if (p.context_lens[b] <= 0) {
          uint4* row = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + size_t(b) * Hq * D);
          for (int i = 0; i < Hq * D * 2 / 16; ++i) row[i] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    const int total = planned ? *reinterpret_cast<volatile int*>(&p.ws.header[kHdrTotal]) : 0;
    const int4* units = reinterpret_cast<const int4*>(p.ws.units);
    const int grp = lane >> 3, gl = lane & 7;
    int it = 0;
    bool first_round = true;
    for (bool more = true; more;) {
      // Keep only a few unclaimed items queued: work left in the global list
      // can still go to whichever CTA frees up first, which keeps the tail short.
      if (planned) {
        const uint64_t t0 = dev::global_timer_ns();
        while (it - *reinterpret_cast<volatile int*>(claim_ctr) > kSchedAhead) {
          if (dev::global_timer_ns() - t0 > tmo) {
            dev::flag_status(p.status, kStatusTimeout);
            return;
          }
          __nanosleep(128);
        }
      }
      PROF_T(t_fetch);
      // The first round is dealt statically (the largest items, one per group
      // and CTA), which saves the counter's round trip at the start; later
      // rounds take the next items from the global counter.
      int idx = total;
      if (planned && gl == 0)
        idx = first_round ? grp * int(gridDim.x) + int(blockIdx.x)
                          : 4 * int(gridDim.x) + atomicAdd(&p.ws.header[kHdrNext], 1);
      first_round = false;
      idx = __shfl_sync(0xffffffffu, idx, grp * 8);
      const bool valid = idx < total;
      int4 u = make_int4(0, 0, 0, 0);
      if (valid) u = units[idx / Hkv];
      const int g = valid ? idx % Hkv : 0;
      const int b = u.x, s = u.y >> 8, nblk = u.y & 0xff, first = u.z, ctx = u.w;
      int phys[kSplitBlocks / 8];
#pragma unroll
      for (int e = 0; e < kSplitBlocks / 8; ++e) {
        const int j = gl + 8 * e;
        phys[e] = 0;
        if (valid && j < nblk) {
          phys[e] = p.block_tables[size_t(b) * p.max_blocks + first + j];
          if (phys[e] < 0 || phys[e] >= p.num_blocks) {
            dev::flag_status(p.status, kStatusBounds);
            phys[e] = 0;
          }
        }
      }
      more = __all_sync(0xffffffffu, valid);
      PROF_ADD(7, t_fetch);
      // push the valid items of this round in group order
      for (int q = 0; q < 4; ++q) {
        if (!__shfl_sync(0xffffffffu, valid, q * 8)) continue;
        const int qs = it % kQueue;
        PROF_T(t_slot);
        if (!mbar_wait_bounded(&item_empty[qs], ((it / kQueue) & 1) ^ 1, tmo, p.status)) return;
        PROF_ADD(8, t_slot);
        if (grp == q) {
          ItemSlot<D>& sl = items[qs];
#pragma unroll
          for (int e = 0; e < kSplitBlocks / 8; ++e) sl.blocks[gl + 8 * e] = phys[e];
          if (gl == 0) {
            const int nblk_all = (ctx + kBlockSize - 1) / kBlockSize;
            sl.b = b;
            sl.g = g;
            sl.s = s;
            sl.ctx = ctx;
            sl.nblk = nblk;
            sl.nsplit = (nblk_all + p.split_blocks - 1) / p.split_blocks;
            sl.first = first;
            const uint32_t qbytes = uint32_t(G) * D * 2;
            dev::mbar_arrive_expect_tx(&item_full[qs], qbytes);
            dev::bulk_load(sl.q,
                           static_cast<const uint8_t*>(p.q) +
                               (size_t(b) * Hq + size_t(g) * G) * D * 2,
                           qbytes, &item_full[qs]);
          } else {
            mbar_arrive(&item_full[qs]);
          }
        }
        ++it;
        __syncwarp();
        if (lane == 0) dev::st_release_cta(pushed, it);
      }
    }
    // no more work: one end marker for each math warp (each takes exactly one)
    for (int e = 0; e < W; ++e, ++it) {
      const int qs = it % kQueue;
      if (!mbar_wait_bounded(&item_empty[qs], ((it / kQueue) & 1) ^ 1, tmo, p.status)) return;
      if (grp == 0) {
        if (gl == 0) items[qs].b = -1;
        mbar_arrive(&item_full[qs]);
      }
      __syncwarp();
      if (lane == 0) dev::st_release_cta(pushed, it + 1);
    }
    if (planned && lane == 0) {
      // The last scheduler to finish returns the work counters to zero, so the
      // next run on this plan starts clean.
      __threadfence();
      if (atomicAdd(&p.ws.header[kHdrDone], 1) == int(gridDim.x) - 1) {
        atomicExch(&p.ws.header[kHdrNext], 0);
        atomicExch(&p.ws.header[kHdrDone], 0);
      }
    }
  } else {
    // -------------------------------------------------------- math warps
    // Each math warp takes whole work items from the queue (in order, one at a
    // time) and streams every block of them through its own small ring,
    // issuing the 2-D tensor copies (128-byte swizzled, L2 evict-first) of a
    // block's K and V tiles NS blocks before it needs them.  Many independent
    // issuers keep HBM busy, and no CTA-wide synchronisation is needed.
    const int w = warp;
    const int n0 = 2 * (lane & 3), n1 = n0 + 1;
    const uint64_t policy = dev::l2_policy_evict_first();
    uint8_t* ring = rings + size_t(w) * NS * S::kStageBytes;
    uint64_t* my_full = full + w * kWarpStages;

    // Waits for item x to be in the queue.  The pushed count goes first: the
    // parity of a queue slot's barrier only tells laps apart once the slot's
    // previous item (x - kQueue) has been pushed, which pushed > x implies.
    auto wait_item = [&](int x) -> bool {
      if (dev::ld_acquire_cta(pushed) <= x) {
        const uint64_t t0 = dev::global_timer_ns();
        while (dev::ld_acquire_cta(pushed) <= x) {
          if (dev::global_timer_ns() - t0 > tmo) {
            dev::flag_status(p.status, kStatusTimeout);
            return false;
          }
          __nanosleep(64);
        }
      }
      return mbar_wait_bounded(&item_full[x % kQueue], (x / kQueue) & 1, tmo, p.status);
    };
    auto claim = [&]() -> int {
      int x = 0;
      if (lane == 0) x = atomicAdd(claim_ctr, 1);
      return __shfl_sync(0xffffffffu, x, 0);
    };
    // items held by this warp, oldest (the one being worked on) first; kept in
    // four registers (h0 is the item in work)
    int h0 = claim(), h1 = 0, h2 = 0, h3 = 0;
    int nheld = 1;
    auto held = [&](int i) { return i == 0 ? h0 : i == 1 ? h1 : i == 2 ? h2 : h3; };
    auto hold = [&](int i, int v) {
      if (i == 1) h1 = v;
      else if (i == 2) h2 = v;
      else if (i == 3) h3 = v;
      else h0 = v;
    };
    // issue cursor: held[ipos], block ij of it; ik blocks issued so far
    int ipos = 0, ij = 0, ik = 0, inblk = -1, ig = 0;
    const ItemSlot<D>* isl = nullptr;
    bool idone = false;
    // Issues this warp's next blocks until NS are in flight.  It never waits
    // for an item whose queue slot this warp itself still holds.
    auto top_up = [&](int kc) -> bool {
      while (!idone && ik < kc + NS) {
        if (inblk < 0) {
          if (ipos == nheld) {
            if (nheld == FIFO) return true;
            hold(nheld++, claim());
          }
          const int x = held(ipos);
          // Lookahead never blocks: an item not in the queue yet is tried again
          // after the next block.  Its block list is readable as soon as it is
          // pushed (release / acquire on the count); only the math needs the
          // query copy to have landed.
          if (x >= h0 + kQueue || dev::ld_acquire_cta(pushed) <= x) return true;
          isl = &items[x % kQueue];
          if (isl->b < 0) {
            idone = true;
            return true;
          }
          inblk = isl->nblk;
          ig = isl->g;
        }
        if (ij >= inblk) {
          ++ipos;
          ij = 0;
          inblk = -1;
          continue;
        }
        const int phys = isl->blocks[ij];
        const int st = ik % NS;
        if (lane == 0) dev::mbar_arrive_expect_tx(&my_full[st], S::kStageBytes);
        __syncwarp();
        // lanes 0..HALVES-1 each issue one 128-byte-wide box of the K tile,
        // then of the V tile (one tensor map per instruction)
        if (lane < HALVES) {
          uint8_t* dst = ring + size_t(st) * S::kStageBytes + lane * 2048;
          const int y = (phys * Hkv + ig) * kBlockSize;
          dev::tma_load_2d(dst, &tmap_k, lane * 64, y, &my_full[st], policy);
          dev::tma_load_2d(dst + S::kTileBytes, &tmap_v, lane * 64, y, &my_full[st], policy);
        }
        ++ik;
        ++ij;
      }
      return true;
    };
    int kc = 0;  // blocks consumed so far
    TIME_MARK(0, dev::global_timer_ns());
    // On a timeout: let this warp's copies in flight land, then give up.
    auto drain = [&]() {
      if (lane == 0)
        for (int k = kc; k < ik; ++k) mbar_wait_bounded(&my_full[k % NS], (k / NS) & 1, tmo, p.status);
      __syncwarp();
    };

    for (;;) {
      const int x = h0;
      const int qs = x % kQueue;
      PROF_T(t_item);
      if (!wait_item(x)) {
        drain();
        return;
      }
      PROF_ADD(3, t_item);
#ifdef PA_PROFILE_TIMES
      if (kc == 0 && (threadIdx.x & 31) == 0 && blockIdx.x * 16 + 15 >= 0)
        g_times[(blockIdx.x * 16 + 14) * 3 + 0 + (warp & 1)] = dev::global_timer_ns();
#endif
      const ItemSlot<D>& sl = items[qs];
      const int b = sl.b;
      if (b < 0) {  // end marker: every block this warp issued has been consumed
        PROF_ADD(11, t_kernel);
        TIME_MARK(1, dev::global_timer_ns());
        TIME_MARK(2, static_cast<unsigned long long>(kc));
        return;
      }
      const int g = sl.g, s = sl.s, ctx = sl.ctx, nblk = sl.nblk, nsplit = sl.nsplit;
      const int first = sl.first;
      // B fragments of Q^T (k = head_dim, n = query head of the group)
      uint32_t qb0[KT], qb1[KT];
      {
        const int hq = lane >> 2;
        const uint16_t* qrow = sl.q + hq * D + n0;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          qb0[kk] = hq < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk) : 0u;
          qb1[kk] = hq < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8) : 0u;
        }
      }
      if (!top_up(kc)) {
        drain();
        return;
      }

      float o[KT][4];
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      const float sl2 = p.scale_log2;

      for (int j = 0; j < nblk; ++j) {
        const int st = kc % NS;
        PROF_T(t_full);
        if (!mbar_wait_bounded(&my_full[st], (kc / NS) & 1, tmo, p.status)) {
          drain();
          return;
        }
        PROF_ADD(0, t_full);
        PROF_T(t_blk);
        const uint32_t kt = dev::smem_u32(ring + size_t(st) * S::kStageBytes);
        const uint32_t vt = kt + S::kTileBytes;
        // ---- S^T (16 tokens x 8 heads) = K (16 x D) . Q^T (D x 8)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int row = lane & 15;
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            const int gc = 2 * kk + (lane >> 4);  // 16-byte chunk along head_dim
            const uint32_t addr =
                kt + (gc >> 3) * 2048 + row * 128 + ((((gc & 7) ^ (row & 7))) << 4);
            uint32_t a0, a1, a2, a3;
            dev::ldmatrix_x4(addr, a0, a1, a2, a3);
            if (kk & 1)
              M::run(sb, a0, a1, a2, a3, qb0[kk], qb1[kk]);
            else
              M::run(sa, a0, a1, a2, a3, qb0[kk], qb1[kk]);
          }
        }
        // ---- mask, scale to base 2, online softmax per head column
        const int valid = ctx - (first + j) * kBlockSize;  // tokens of the block in context
        const int r0 = lane >> 2;
        const bool v0 = r0 < valid, v1 = r0 + 8 < valid;
        const float x0 = v0 ? (sa[0] + sb[0]) * sl2 : -INFINITY;
        const float x1 = v0 ? (sa[1] + sb[1]) * sl2 : -INFINITY;
        const float x2 = v1 ? (sa[2] + sb[2]) * sl2 : -INFINITY;
        const float x3 = v1 ? (sa[3] + sb[3]) * sl2 : -INFINITY;
        float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o_));
          bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o_));
        }
        const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
        const float al0 = dev::fast_exp2(m0 - mn0), al1 = dev::fast_exp2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const uint32_t p01 = M::pack(dev::fast_exp2(x0 - mn0), dev::fast_exp2(x1 - mn1));
        const uint32_t p23 = M::pack(dev::fast_exp2(x2 - mn0), dev::fast_exp2(x3 - mn1));
        {
          const float2 f01 = M::unpack(p01), f23 = M::unpack(p23);
          l0 = l0 * al0 + f01.x + f23.x;
          l1 = l1 * al1 + f01.y + f23.y;
        }
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
        // ---- P^T as the B operand: transpose the two 8x8 halves in registers
        const uint32_t pb0 = dev::movmatrix_trans(p01);
        const uint32_t pb1 = dev::movmatrix_trans(p23);
        // V^T fragments hold tokens 2(lane%4)+{0,1} (a0, a1) and +8 (a2, a3):
        // zero the ones past the context so their bits never meet P = 0.
        uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
        if (valid < kBlockSize) {
          const int t = 2 * (lane & 3);
          vm_lo = (t < valid ? 0x0000ffffu : 0u) | (t + 1 < valid ? 0xffff0000u : 0u);
          vm_hi = (t + 8 < valid ? 0x0000ffffu : 0u) | (t + 9 < valid ? 0xffff0000u : 0u);
        }
        // ---- O^T (D x 8) += V^T (D x 16 tokens) . P^T (16 tokens x 8)
        {
          const int tok = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            const int gc = 2 * mt + ((lane >> 3) & 1);
            const uint32_t addr =
                vt + (gc >> 3) * 2048 + tok * 128 + ((((gc & 7) ^ (tok & 7))) << 4);
            uint32_t a0, a1, a2, a3;
            dev::ldmatrix_x4_trans(addr, a0, a1, a2, a3);
            M::run(o[mt], a0 & vm_lo, a1 & vm_lo, a2 & vm_hi, a3 & vm_hi, pb0, pb1);
          }
        }
        // the stage is read; order those reads before the copy that reuses it
        dev::fence_proxy_async_smem();
        __syncwarp();
        ++kc;
        PROF_ADD(1, t_blk);
        PROF_INC(9, 1);
        PROF_T(t_issue);
        if (!top_up(kc)) {
          drain();
          return;
        }
        PROF_ADD(4, t_issue);
      }
      PROF_T(t_end);
      PROF_INC(10, 1);

      // ---- end of the item: this warp holds the whole (m, l, O) of its split
#pragma unroll
      for (int o_ = 4; o_ < 32; o_ <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
      }
      const float inv0 = 1.f / l0, inv1 = 1.f / l1;
      const size_t head0 = size_t(b) * Hq + size_t(g) * G;
      if (nsplit == 1) {
        T* orow = static_cast<T*>(p.out) + head0 * D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          const int d0 = 16 * mt + (lane >> 2);
          if (n0 < G) {
            orow[n0 * D + d0] = M::from_float(o[mt][0] * inv0);
            orow[n0 * D + d0 + 8] = M::from_float(o[mt][2] * inv0);
          }
          if (n1 < G) {
            orow[n1 * D + d0] = M::from_float(o[mt][1] * inv1);
            orow[n1 * D + d0 + 8] = M::from_float(o[mt][3] * inv1);
          }
        }
      } else {
        const size_t part0 = (size_t(b) * p.max_splits + s) * Hq + size_t(g) * G;
        float* prow = p.ws.part_o + part0 * D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          const int d0 = 16 * mt + (lane >> 2);
          if (n0 < G) {
            prow[n0 * D + d0] = o[mt][0] * inv0;
            prow[n0 * D + d0 + 8] = o[mt][2] * inv0;
          }
          if (n1 < G) {
            prow[n1 * D + d0] = o[mt][1] * inv1;
            prow[n1 * D + d0 + 8] = o[mt][3] * inv1;
          }
        }
        if (lane < 4) {
          if (n0 < G) p.ws.part_lse[part0 + n0] = m0 + log2f(l0);
          if (n1 < G) p.ws.part_lse[part0 + n1] = m1 + log2f(l1);
        }
        // publish this split, count it; the warp that completes (b, g) merges
        __threadfence();
        int last = 0;
        if (lane == 0)
          last = atomicAdd(&p.ws.arrivals[size_t(b) * Hkv + g], 1) == nsplit - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const size_t pbase = size_t(b) * p.max_splits * Hq + size_t(g) * G;
          T* orow = static_cast<T*>(p.out) + head0 * D;
          // each lane owns 4 consecutive outputs per pass (one float4 per split)
          for (int c = lane; c < G * D / 4; c += 32) {
            const int hh = (c * 4) / D, dd = (c * 4) % D;
            float mrun = -INFINITY, lrun = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int sp = 0; sp < nsplit; ++sp) {
              const size_t r = pbase + size_t(sp) * Hq + hh;
              const float lse = __ldcg(&p.ws.part_lse[r]);
              const float4 ov = __ldcg(reinterpret_cast<const float4*>(&p.ws.part_o[r * D + dd]));
              const float mn = fmaxf(mrun, lse);
              const float a = dev::fast_exp2(mrun - mn), wv = dev::fast_exp2(lse - mn);
              acc.x = acc.x * a + wv * ov.x;
              acc.y = acc.y * a + wv * ov.y;
              acc.z = acc.z * a + wv * ov.z;
              acc.w = acc.w * a + wv * ov.w;
              lrun = lrun * a + wv;
              mrun = mn;
            }
            const float inv = 1.f / lrun;
            orow[hh * D + dd + 0] = M::from_float(acc.x * inv);
            orow[hh * D + dd + 1] = M::from_float(acc.y * inv);
            orow[hh * D + dd + 2] = M::from_float(acc.z * inv);
            orow[hh * D + dd + 3] = M::from_float(acc.w * inv);
          }
          if (lane == 0) p.ws.arrivals[size_t(b) * Hkv + g] = 0;  // ready for the next run
        }
      }
      // done with this item: free its queue slot, move to the next one
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[qs]);
      h0 = h1;
      h1 = h2;
      h2 = h3;
      --nheld;
      --ipos;
      if (nheld == 0) {
        h0 = claim();
        nheld = 1;
        ipos = 0;
      }
      PROF_ADD(2, t_end);
    }
  }
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
  int split_blocks = 0;  // 0: by group size (16 blocks for G == 1, 32 otherwise)
  int warps = kConsumerWarps;
  int ctas_per_sm = 1;
  int max_stages = kWarpStages;
};
Tuning read_tuning_env() {
  Tuning t;
  if (const char* v = std::getenv("PA_DECODE_WARPS")) t.warps = std::atoi(v) == 4 ? 4 : 8;
  if (const char* v = std::getenv("PA_DECODE_SPLIT_BLOCKS"))
    t.split_blocks = std::max(kMinSplitBlocks, std::min(kSplitBlocks, std::atoi(v)));
  if (const char* v = std::getenv("PA_DECODE_CTAS_PER_SM")) t.ctas_per_sm = std::max(1, std::min(4, std::atoi(v)));
  if (const char* v = std::getenv("PA_DECODE_MAX_STAGES")) t.max_stages = std::max(1, std::min(kWarpStages, std::atoi(v)));
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
  KernelConfig cfg[2][2][kMaxGroup + 1];  // [bf16?][head_dim 128?][group]
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <typename T, int D, int W>
cudaError_t configure_kernel(KernelConfig* cfg, const Tuning& t, size_t optin, size_t per_sm) {
  // shared memory per CTA when `ctas_per_sm` CTAs share an SM (1 KiB reserved each)
  size_t budget = per_sm / t.ctas_per_sm - 1024;
  if (budget > optin) budget = optin;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, W>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(budget));
  for (int g = 1; g <= kMaxGroup && e == cudaSuccess; ++g) {
    int stages = Smem<D, W>::stages_for(g, budget);  // per math warp
    if (stages > t.max_stages) stages = t.max_stages;
    cfg[g].stages = stages;
    cfg[g].smem = Smem<D, W>::bytes(g, stages);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cfg[g].ctas_per_sm, decode_kernel<T, D, W>,
                                                      (W + 1) * 32, cfg[g].smem);
    if (cfg[g].ctas_per_sm > t.ctas_per_sm) cfg[g].ctas_per_sm = t.ctas_per_sm;
  }
  return e;
}

template <int W>
cudaError_t configure_all(DeviceState& st, size_t optin, size_t per_sm) {
  cudaError_t e = configure_kernel<__nv_bfloat16, 128, W>(st.cfg[1][1], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__nv_bfloat16, 64, W>(st.cfg[1][0], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__half, 128, W>(st.cfg[0][1], st.tuning, optin, per_sm);
  if (e == cudaSuccess) e = configure_kernel<__half, 64, W>(st.cfg[0][0], st.tuning, optin, per_sm);
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
        for (int g = 1; g <= kMaxGroup; ++g)
          if (st.cfg[a][d][g].stages < 1 || st.cfg[a][d][g].ctas_per_sm < 1)
            st.error = PA_ERR_UNSUPPORTED;
  });
  if (st.error != PA_OK) return fail(st.error, "decode: per-device set-up failed on device %d", device);
  return PA_OK;
}

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(PA_ERR_CUDA, "decode: cuTensorMapEncodeTiled is unavailable");
  return PA_OK;
}

// 2-D view of a cache: rows = num_blocks * num_kv_heads * 16 token rows of
// head_dim elements; one copy box = 16 rows x 64 elements (128 bytes wide,
// 128-byte swizzle), so a (block, head) tile is head_dim / 64 boxes.  In
// shared memory, box h of a tile sits at h * 2048, row r at r * 128, with its
// 16-byte chunks XOR-swizzled by r % 8.
int encode_cache_map(CUtensorMap* map, const void* cache, bool bf16, int num_blocks,
                     int num_kv_heads, int head_dim) {
  const cuuint64_t dims[2] = {cuuint64_t(head_dim),
                              cuuint64_t(num_blocks) * num_kv_heads * kBlockSize};
  const cuuint64_t strides[1] = {cuuint64_t(head_dim) * 2};
  const cuuint32_t box[2] = {64, kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(cache), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed (%d)", int(r));
  return PA_OK;
}

// Per-thread cache of encoded tensor maps: a decode step reuses the same layer
// caches every step, and encoding is a host-side driver call.
struct MapKey {
  const void* ptr;
  int num_blocks, num_kv_heads, head_dim;
  bool bf16;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && num_blocks == o.num_blocks && num_kv_heads == o.num_kv_heads &&
           head_dim == o.head_dim && bf16 == o.bf16;
  }
};
struct MapEntry {
  MapKey key{nullptr, 0, 0, 0, false};
  alignas(64) CUtensorMap map;
};
constexpr int kMapCache = 256;
thread_local MapEntry t_maps[kMapCache];

int cached_cache_map(CUtensorMap* out, const void* cache, bool bf16, int num_blocks,
                     int num_kv_heads, int head_dim) {
  const MapKey key{cache, num_blocks, num_kv_heads, head_dim, bf16};
  uint64_t h = reinterpret_cast<uintptr_t>(cache) >> 8;
  h ^= uint64_t(num_blocks) * 0x9E3779B97F4A7C15ull ^ uint64_t(num_kv_heads * 131 + head_dim);
  MapEntry& e = t_maps[(h ^ (h >> 17)) % kMapCache];
  if (!(e.key == key)) {
    int rc = encode_cache_map(&e.map, cache, bf16, num_blocks, num_kv_heads, head_dim);
    if (rc != PA_OK) {
      e.key = MapKey{nullptr, 0, 0, 0, false};
      return rc;
    }
    e.key = key;
  }
  *out = e.map;
  return PA_OK;
}

template <typename T, int D, int W>
int launch_tc(Params prm, const KernelConfig& kc, int sms, cudaStream_t stream) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  alignas(64) CUtensorMap mk, mv;
  int rc = cached_cache_map(&mk, prm.k_cache, kBf16, prm.num_blocks, prm.num_kv_heads, D);
  if (rc == PA_OK) rc = cached_cache_map(&mv, prm.v_cache, kBf16, prm.num_blocks, prm.num_kv_heads, D);
  if (rc != PA_OK) return rc;
  prm.stages = kc.stages;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms * kc.ctas_per_sm);
  cfg.blockDim = dim3((W + 1) * 32);
  cfg.dynamicSmemBytes = kc.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<T, D, W>, mk, mv, prm);
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
  prm.split_blocks = tuning().split_blocks
                         ? tuning().split_blocks
                         : (num_q_heads == num_kv_heads ? kMinSplitBlocks : kSplitBlocks);
  prm.signature = plan_signature(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                 prm.split_blocks);
  prm.ws.header = reinterpret_cast<int*>(ws + lay.header);
  prm.ws.units = reinterpret_cast<int*>(ws + lay.units);
  prm.ws.arrivals = reinterpret_cast<int*>(ws + lay.arrivals);
  prm.ws.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  prm.ws.part_o = reinterpret_cast<float*>(ws + lay.part_o);
  prm.status = status;
  prm.timeout_ns = 1000000000ull;  // 1 s per wait
  return prm;
}

int plan_impl(const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
              int head_dim, int max_blocks_per_seq, void* workspace, size_t workspace_bytes,
              cudaStream_t stream, const char* who) {
  const Layout lay =
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  int rc = check_workspace(workspace, workspace_bytes, lay, who);
  if (rc != PA_OK) return rc;
  if (!context_lens) return fail(PA_ERR_INVALID_ARG, "%s: context_lens is NULL", who);
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  const Params prm = make_params(context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 max_blocks_per_seq, workspace, lay, status);
  static std::once_flag carveout_once;
  std::call_once(carveout_once, [] {
    // keep the SM's shared-memory split the attention kernel wants, so no
    // reconfiguration happens between the plan and the attention kernel
    cudaFuncSetAttribute(plan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
  });
  plan_kernel<<<1, 1024, 0, stream>>>(prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: plan launch failed: %s", who, cudaGetErrorString(e));
  return PA_OK;
}

int run_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
             const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
             int head_dim, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
             void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream,
             const char* who) {
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "%s: num_blocks must be positive", who);
  if (double(num_blocks) * num_kv_heads * kBlockSize >= 2147483647.0)
    return fail(PA_ERR_INVALID_ARG, "%s: cache has too many rows", who);
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", who);
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out))
    return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", who);
  const Layout lay =
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  int rc = check_workspace(workspace, workspace_bytes, lay, who);
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
  rc = get_encoder();
  if (rc != PA_OK) return rc;
  const DeviceState& st = g_dev[device];
  const KernelConfig& kc = st.cfg[dtype == PA_BF16][head_dim == 128][prm.group];
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

#ifdef PA_PROFILE
// Copies (and clears) the per-CTA cycle counters of a -DPA_PROFILE build.
PA_API int pa_profile_read(unsigned long long* host, int ctas) {
  const size_t bytes = size_t(ctas) * kProfSlots * sizeof(unsigned long long);
  if (cudaMemcpyFromSymbol(host, g_prof, bytes) != cudaSuccess) return PA_ERR_CUDA;
  static unsigned long long zeros[2048 * kProfSlots];
  if (cudaMemcpyToSymbol(g_prof, zeros, bytes) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}
#endif

#ifdef PA_PROFILE_TIMES
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
  *bytes = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq).total;
  return PA_OK;
}

PA_API int pa_paged_attention_decode_plan(const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq, void* workspace,
                                          size_t workspace_bytes, void* stream) {
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
  const char* who = "paged_attention_decode_run";
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  return run_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype, out,
                  workspace, workspace_bytes, static_cast<cudaStream_t>(stream), who);
}

PA_API int pa_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                     void* out, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  const char* who = "paged_attention_decode";
  int rc = check_decode_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               dtype, who);
  if (rc != PA_OK || num_seqs == 0) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
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

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB per device
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
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode_noalloc: sizes must be positive");
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
