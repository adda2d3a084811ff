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
//    the tail of the persistent kernel is made of the smallest items.
//  * persistent attention kernel, one or two CTAs per SM, three warp roles:
//      - scheduler warp: takes the next item from a global counter, reads the
//        item's block-table entries (range-checked) and bulk-copies the G
//        query rows of (b, g) into a shared-memory item queue;
//      - TMA warp: for every block of the item issues 2-D tensor copies of the
//        16 x head_dim K tile and V tile (each a contiguous 2 or 4 KiB run of
//        the cache) into a ring of kStages shared-memory stages, 128-byte
//        swizzled, with L2 evict-first hints (the cache is streamed once);
//      - kConsumerWarps math warps: warp w takes blocks w, w+W, ... of the
//        item.  Per 16-token block: S^T = K . Q^T on the tensor cores
//        (m16n8k16, M = the 16 tokens, N = the G <= 8 query heads of the
//        group, K = head_dim), online softmax in base 2 with per-head running
//        max / sum, P rounded to the input type and transposed in registers
//        (movmatrix), O^T += V^T . P^T (M = head_dim rows of V^T via
//        ldmatrix.trans).  Each K/V tile is read from HBM once for the whole
//        query group.
//    At the end of an item the math warps merge their partial (m, l, O)
//    through shared memory.  A sequence with one split writes `out`
//    directly; otherwise the item writes (o, lse) to the workspace and the
//    CTA that finishes the last split of (b, g) merges all splits with
//    log-sum-exp weights (an arrival counter, no spinning).
//  * Every wait is an mbarrier wait with a time limit; running out sets the
//    timeout bit of the device status word and the warp returns.
//
// An fp32 path (CUDA cores, one warp per (sequence, head), online softmax in
// natural base) serves float32 caches; it is exact to fp32 rounding and is not
// tuned for speed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <cstring>
#include <mutex>

#include "decode.cuh"
#include "device_common.cuh"
#include "pagedattn.h"
#include "status.h"

namespace pa {
namespace decode {

using dev::mbar_arrive;
using dev::mbar_wait_bounded;

template <int D>
struct alignas(128) ItemSlot {
  int b, g, s, ctx, nblk, nsplit, pad0, pad1;
  int blocks[kSplitBlocks];
  alignas(16) uint16_t q[kMaxGroup * D];
};

template <int D>
struct Smem {
  static constexpr int kTileBytes = kBlockSize * D * 2;  // one (block, head) tile
  static constexpr int kStageBytes = 2 * kTileBytes;     // K tile + V tile
  static constexpr size_t kRing = size_t(kStages) * kStageBytes;
  static constexpr size_t kItems = size_t(kQueue) * sizeof(ItemSlot<D>);
  static constexpr int kOPitch = D + 4;                  // floats; breaks bank conflicts
  __host__ __device__ static size_t merge_o_floats(int group) { return size_t(2) * kConsumerWarps * group * kOPitch; }
  static constexpr size_t kMergeMl = size_t(2) * kConsumerWarps * kMaxGroup * 2;  // floats
  static constexpr size_t kBars = 2 * kStages + 2 * kQueue + 3;                   // uint64
  static size_t bytes(int group) {
    return 1024 /* alignment slack */ + kRing + kItems + merge_o_floats(group) * 4 +
           kMergeMl * 4 + kBars * 8 + 16;
  }
};

// ------------------------------------------------------------------ plan
__global__ void __launch_bounds__(1024) plan_kernel(const Params p, int out_row_vecs) {
  __shared__ int hist[kSplitBlocks];
  __shared__ int bucket[kSplitBlocks];
  __shared__ int warp_tot[32];
  __shared__ int carry;
  dev::grid_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kSplitBlocks) hist[tid] = 0;
  if (tid == 0) carry = 0;
  __syncthreads();
  const int cap = p.max_blocks * kBlockSize;
  int4* units = reinterpret_cast<int4*>(p.ws.units);

  for (int base = 0; base < p.num_seqs; base += 1024) {
    const int b = base + tid;
    int nfull = 0, ctx = 0;
    if (b < p.num_seqs) {
      ctx = p.context_lens[b];
      if (ctx < 0 || ctx > cap) {
        dev::flag_status(p.status, kStatusBounds);
        ctx = ctx < 0 ? 0 : cap;
      }
      const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
      nfull = nblk / kSplitBlocks;
      const int rem = nblk % kSplitBlocks;
      if (rem) atomicAdd(&hist[rem], 1);
      for (int g = 0; g < p.num_kv_heads; ++g) p.ws.arrivals[size_t(b) * p.num_kv_heads + g] = 0;
      if (ctx == 0) {  // empty context: zero output row
        uint4* row = reinterpret_cast<uint4*>(p.out) + size_t(b) * out_row_vecs;
        for (int i = 0; i < out_row_vecs; ++i) row[i] = make_uint4(0, 0, 0, 0);
      }
    }
    // block-wide exclusive scan of nfull
    int incl = nfull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane], ti = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, ti, o);
        if (lane >= o) ti += y;
      }
      warp_tot[lane] = ti - t;
    }
    __syncthreads();
    const int excl = carry + warp_tot[warp] + incl - nfull;
    for (int k = 0; k < nfull; ++k) units[excl + k] = make_int4(b, k, ctx, kSplitBlocks);
    __syncthreads();
    if (tid == 1023) carry = excl + nfull;
    __syncthreads();
  }
  if (tid == 0) {
    int pos = carry;
    for (int r = kSplitBlocks - 1; r >= 1; --r) {
      bucket[r] = pos;
      pos += hist[r];
    }
    p.ws.header[1] = pos * p.num_kv_heads;
    p.ws.header[0] = 0;
  }
  __syncthreads();
  for (int b = tid; b < p.num_seqs; b += 1024) {
    int ctx = p.context_lens[b];
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
    const int rem = nblk % kSplitBlocks;
    if (rem) {
      const int pos = atomicAdd(&bucket[rem], 1);
      units[pos] = make_int4(b, nblk / kSplitBlocks, ctx, rem);
    }
  }
}

// --------------------------------------------------------- tensor-core path
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                          const __grid_constant__ CUtensorMap tmap_v,
                                                          const Params p) {
  using S = Smem<D>;
  using M = dev::Mma<T>;
  constexpr int W = kConsumerWarps;
  constexpr int KT = D / 16;  // 16-wide steps along head_dim
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int G = p.group;
  uint8_t* ring = smem;
  ItemSlot<D>* items = reinterpret_cast<ItemSlot<D>*>(ring + S::kRing);
  float* merge_o = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(items) + S::kItems);
  float* merge_ml = merge_o + S::merge_o_floats(G);
  uint64_t* full = reinterpret_cast<uint64_t*>(merge_ml + S::kMergeMl);
  uint64_t* empty = full + kStages;
  uint64_t* item_full = empty + kStages;
  uint64_t* item_empty = item_full + kQueue;
  uint64_t* mb_merge = item_empty + kQueue;
  uint64_t* mb_fence = mb_merge + 1;
  uint64_t* mb_flag = mb_fence + 1;
  volatile int* last_flag = reinterpret_cast<volatile int*>(mb_flag + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      dev::mbar_init(&full[i], 1);
      dev::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kQueue; ++i) {
      dev::mbar_init(&item_full[i], 32);
      dev::mbar_init(&item_empty[i], W + 1);
    }
    dev::mbar_init(mb_merge, W * 32);
    dev::mbar_init(mb_fence, W * 32);
    dev::mbar_init(mb_flag, 1);
    dev::mbar_fence_init();
  }
  if (warp == W) {
    dev::prefetch_tensormap(&tmap_k);
    dev::prefetch_tensormap(&tmap_v);
  }
  __syncthreads();
  dev::grid_dependency_wait();  // the plan kernel's work list is complete

  const unsigned long long tmo = p.timeout_ns;
  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;

  if (warp == W + 1) {
    // ------------------------------------------------------------ scheduler
    const int total = *reinterpret_cast<volatile int*>(&p.ws.header[1]);
    const int4* units = reinterpret_cast<const int4*>(p.ws.units);
    for (int it = 0;; ++it) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(&p.ws.header[0], 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      const int qs = it % kQueue;
      if (!mbar_wait_bounded(&item_empty[qs], ((it / kQueue) & 1) ^ 1, tmo, p.status)) return;
      ItemSlot<D>& sl = items[qs];
      if (idx >= total) {
        if (lane == 0) sl.b = -1;
        mbar_arrive(&item_full[qs]);
        return;
      }
      const int4 u = units[idx / Hkv];
      const int g = idx % Hkv;
      const int b = u.x, s = u.y, ctx = u.z, nblk = u.w;
      int phys = 0;
      if (lane < nblk) {
        phys = p.block_tables[size_t(b) * p.max_blocks + s * kSplitBlocks + lane];
        if (phys < 0 || phys >= p.num_blocks) {
          dev::flag_status(p.status, kStatusBounds);
          phys = 0;
        }
      }
      sl.blocks[lane] = phys;
      if (lane == 0) {
        const int nblk_all = (ctx + kBlockSize - 1) / kBlockSize;
        sl.b = b;
        sl.g = g;
        sl.s = s;
        sl.ctx = ctx;
        sl.nblk = nblk;
        sl.nsplit = (nblk_all + kSplitBlocks - 1) / kSplitBlocks;
        const uint32_t qbytes = uint32_t(G) * D * 2;
        dev::mbar_arrive_expect_tx(&item_full[qs], qbytes);
        dev::bulk_load(sl.q,
                       static_cast<const uint8_t*>(p.q) + (size_t(b) * Hq + size_t(g) * G) * D * 2,
                       qbytes, &item_full[qs]);
      } else {
        mbar_arrive(&item_full[qs]);
      }
    }
  } else if (warp == W) {
    // ---------------------------------------------------------- TMA issuer
    const uint64_t policy = dev::l2_policy_evict_first();
    int n = 0;
    for (int it = 0;; ++it) {
      const int qs = it % kQueue;
      if (!mbar_wait_bounded(&item_full[qs], (it / kQueue) & 1, tmo, p.status)) return;
      const ItemSlot<D>& sl = items[qs];
      const int b = sl.b;
      const int nblk = b < 0 ? 0 : sl.nblk;
      const int g = sl.g;
      const int my_phys = sl.blocks[lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[qs]);
      if (b < 0) return;
      for (int j = 0; j < nblk; ++j, ++n) {
        const int phys = __shfl_sync(0xffffffffu, my_phys, j);
        if (lane == 0) {
          const int st = n % kStages;
          if (!mbar_wait_bounded(&empty[st], ((n / kStages) & 1) ^ 1, tmo, p.status)) {
            // Let the copies already issued land before the CTA exits.
            for (int k = 1; k <= kStages && n - k >= 0; ++k) {
              const int m = n - k;
              mbar_wait_bounded(&full[m % kStages], (m / kStages) & 1, tmo, p.status);
            }
            n = -1;
          } else {
            dev::mbar_arrive_expect_tx(&full[st], S::kStageBytes);
            uint8_t* stage = ring + size_t(st) * S::kStageBytes;
            const int y = (phys * Hkv + g) * kBlockSize;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              dev::tma_load_2d(stage + h * 2048, &tmap_k, h * 64, y, &full[st], policy);
              dev::tma_load_2d(stage + S::kTileBytes + h * 2048, &tmap_v, h * 64, y, &full[st],
                               policy);
            }
          }
        }
        n = __shfl_sync(0xffffffffu, n, 0);
        if (n < 0) return;
      }
    }
  } else {
    // -------------------------------------------------------- math warps
    const int w = warp;
    const int tid = threadIdx.x;  // 0 .. W*32-1
    const int n0 = 2 * (lane & 3), n1 = n0 + 1;
    uint32_t merge_phase = 0, fence_phase = 0, flag_phase = 0;
    int n_base = 0;
    for (int it = 0;; ++it) {
      const int qs = it % kQueue;
      if (!mbar_wait_bounded(&item_full[qs], (it / kQueue) & 1, tmo, p.status)) return;
      const ItemSlot<D>& sl = items[qs];
      const int b = sl.b;
      if (b < 0) return;
      const int g = sl.g, s = sl.s, ctx = sl.ctx, nblk = sl.nblk, nsplit = sl.nsplit;
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[qs]);

      float o[KT][4];
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      const float sl2 = p.scale_log2;

      for (int j = w; j < nblk; j += W) {
        const int nn = n_base + j;
        const int st = nn % kStages;
        if (!mbar_wait_bounded(&full[st], (nn / kStages) & 1, tmo, p.status)) return;
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
        const int tok0 = (s * kSplitBlocks + j) * kBlockSize + (lane >> 2);
        const bool v0 = tok0 < ctx, v1 = tok0 + 8 < ctx;
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
            M::run(o[mt], a0, a1, a2, a3, pb0, pb1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      n_base += nblk;

      // ---- merge the W warps' partial states through shared memory
#pragma unroll
      for (int o_ = 4; o_ < 32; o_ <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
      }
      const int pb = it & 1;
      float* ow = merge_o + (size_t(pb) * W + w) * G * S::kOPitch;
      float* mlw = merge_ml + (size_t(pb) * W + w) * kMaxGroup * 2;
      if (lane < 4) {
        if (n0 < G) {
          mlw[n0 * 2] = m0;
          mlw[n0 * 2 + 1] = l0;
        }
        if (n1 < G) {
          mlw[n1 * 2] = m1;
          mlw[n1 * 2 + 1] = l1;
        }
      }
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        const int d0 = 16 * mt + (lane >> 2);
        if (n0 < G) {
          ow[n0 * S::kOPitch + d0] = o[mt][0];
          ow[n0 * S::kOPitch + d0 + 8] = o[mt][2];
        }
        if (n1 < G) {
          ow[n1 * S::kOPitch + d0] = o[mt][1];
          ow[n1 * S::kOPitch + d0 + 8] = o[mt][3];
        }
      }
      mbar_arrive(mb_merge);
      if (!mbar_wait_bounded(mb_merge, merge_phase, tmo, p.status)) return;
      merge_phase ^= 1;

      const float* obuf = merge_o + size_t(pb) * W * G * S::kOPitch;
      const float* mlbuf = merge_ml + size_t(pb) * W * kMaxGroup * 2;
      const size_t head0 = size_t(b) * Hq + size_t(g) * G;
      const size_t part0 = (size_t(b) * p.max_splits + s) * Hq + size_t(g) * G;
      for (int e = tid; e < G * D; e += W * 32) {
        const int hh = e / D, dd = e - hh * D;
        float mf = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < W; ++ww) mf = fmaxf(mf, mlbuf[ww * kMaxGroup * 2 + hh * 2]);
        float acc = 0.f, ls = 0.f;
#pragma unroll
        for (int ww = 0; ww < W; ++ww) {
          const float wt = dev::fast_exp2(mlbuf[ww * kMaxGroup * 2 + hh * 2] - mf);
          acc += wt * obuf[(ww * G + hh) * S::kOPitch + dd];
          ls += wt * mlbuf[ww * kMaxGroup * 2 + hh * 2 + 1];
        }
        const float val = acc / ls;
        if (nsplit == 1) {
          static_cast<T*>(p.out)[(head0 + hh) * D + dd] = M::from_float(val);
        } else {
          p.ws.part_o[(part0 + hh) * D + dd] = val;
          if (dd == 0) p.ws.part_lse[part0 + hh] = mf + log2f(ls);
        }
      }
      if (nsplit > 1) {
        // ---- the CTA finishing the last split of (b, g) merges all splits
        __threadfence();
        mbar_arrive(mb_fence);
        if (!mbar_wait_bounded(mb_fence, fence_phase, tmo, p.status)) return;
        fence_phase ^= 1;
        if (tid == 0) {
          const int old = atomicAdd(&p.ws.arrivals[size_t(b) * Hkv + g], 1);
          *last_flag = (old == nsplit - 1);
          __threadfence();
          mbar_arrive(mb_flag);
        }
        if (!mbar_wait_bounded(mb_flag, flag_phase, tmo, p.status)) return;
        flag_phase ^= 1;
        if (*last_flag) {
          __threadfence();
          const size_t pbase = size_t(b) * p.max_splits * Hq + size_t(g) * G;
          for (int e = tid; e < G * D; e += W * 32) {
            const int hh = e / D, dd = e - hh * D;
            float mrun = -INFINITY, lrun = 0.f, acc = 0.f;
            for (int sp = 0; sp < nsplit; ++sp) {
              const size_t r = pbase + size_t(sp) * Hq + hh;
              const float lse = __ldcg(&p.ws.part_lse[r]);
              const float ov = __ldcg(&p.ws.part_o[r * D + dd]);
              const float mn = fmaxf(mrun, lse);
              const float a = dev::fast_exp2(mrun - mn), wv = dev::fast_exp2(lse - mn);
              acc = acc * a + wv * ov;
              lrun = lrun * a + wv;
              mrun = mn;
            }
            static_cast<T*>(p.out)[(head0 + hh) * D + dd] = M::from_float(acc / lrun);
          }
        }
      }
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

struct DeviceState {
  std::once_flag once;
  int error = 0;  // PA_OK or the status the set-up failed with
  int sms = 0;
  int ctas_per_sm[2][2][kMaxGroup + 1] = {};  // [bf16?][head_dim 128?][group]
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <typename T, int D>
cudaError_t configure_kernel(int* ctas) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Smem<D>::bytes(kMaxGroup)));
  for (int g = 1; g <= kMaxGroup && e == cudaSuccess; ++g)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas[g], decode_kernel<T, D>, kThreads,
                                                      Smem<D>::bytes(g));
  return e;
}

int device_setup(int device) {
  DeviceState& st = g_dev[device];
  std::call_once(st.once, [&] {
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      st.error = PA_ERR_CUDA;
      return;
    }
    cudaError_t e = configure_kernel<__nv_bfloat16, 128>(st.ctas_per_sm[1][1]);
    if (e == cudaSuccess) e = configure_kernel<__nv_bfloat16, 64>(st.ctas_per_sm[1][0]);
    if (e == cudaSuccess) e = configure_kernel<__half, 128>(st.ctas_per_sm[0][1]);
    if (e == cudaSuccess) e = configure_kernel<__half, 64>(st.ctas_per_sm[0][0]);
    st.error = e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
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
// 128-byte swizzle).
int encode_cache_map(CUtensorMap* map, const void* cache, int dtype, int num_blocks,
                     int num_kv_heads, int head_dim) {
  const cuuint64_t dims[2] = {cuuint64_t(head_dim),
                              cuuint64_t(num_blocks) * num_kv_heads * kBlockSize};
  const cuuint64_t strides[1] = {cuuint64_t(head_dim) * 2};
  const cuuint32_t box[2] = {64, kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(cache), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed (%d)", int(r));
  return PA_OK;
}

template <typename T, int D>
int launch_tc(const Params& prm, const void* k_cache, const void* v_cache, int dtype,
              cudaStream_t stream, int grid) {
  alignas(64) CUtensorMap mk, mv;
  int rc = encode_cache_map(&mk, k_cache, dtype, prm.num_blocks, prm.num_kv_heads, D);
  if (rc == PA_OK) rc = encode_cache_map(&mv, v_cache, dtype, prm.num_blocks, prm.num_kv_heads, D);
  if (rc != PA_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<D>::bytes(prm.group);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<T, D>, mk, mv, prm);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "decode: launch failed: %s", cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace
}  // namespace decode
}  // namespace pa

using namespace pa;
using namespace pa::decode;

extern "C" {

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

PA_API int pa_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                     void* out, void* workspace, size_t workspace_bytes,
                                     void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "paged_attention_decode: unknown dtype %d", dtype);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "paged_attention_decode: head_dim %d (64 or 128)", head_dim);
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode: sizes must be positive");
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode: num_q_heads %% num_kv_heads != 0");
  const int group = num_q_heads / num_kv_heads;
  if (dtype != PA_F32 && group > kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "paged_attention_decode: %d query heads per KV head (max %d)",
                group, kMaxGroup);
  if (double(num_blocks) * num_kv_heads * kBlockSize >= 2147483647.0)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode: cache has too many rows");
  if (double(max_blocks_per_seq) * kBlockSize >= 2147483647.0)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode: max_blocks_per_seq too large");
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode: NULL pointer");
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(PA_ERR_INVALID_ARG,
                "paged_attention_decode: tensors must be 16-byte aligned, workspace 256-byte");
  const Layout lay =
      workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
  if (workspace_bytes < lay.total)
    return fail(PA_ERR_INVALID_ARG, "paged_attention_decode: workspace %zu bytes < %zu needed",
                workspace_bytes, lay.total);

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device >= kMaxDevices)
    return fail(PA_ERR_CUDA, "paged_attention_decode: no current CUDA device");
  int rc = device_setup(device);
  if (rc != PA_OK) return rc;
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Params prm = {};
  prm.q = q;
  prm.k_cache = k_cache;
  prm.v_cache = v_cache;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = group;
  prm.head_dim = head_dim;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = num_blocks;
  prm.max_splits = lay.max_splits;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.ws.header = reinterpret_cast<int*>(ws + lay.header);
  prm.ws.units = reinterpret_cast<int*>(ws + lay.units);
  prm.ws.arrivals = reinterpret_cast<int*>(ws + lay.arrivals);
  prm.ws.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  prm.ws.part_o = reinterpret_cast<float*>(ws + lay.part_o);
  prm.status = status;
  prm.timeout_ns = 1000000000ull;  // 1 s per wait

  if (dtype == PA_F32) {
    const int warps = num_seqs * num_q_heads;
    const int blocks = (warps + 3) / 4;
    if (head_dim == 64)
      decode_f32_kernel<64><<<blocks, 128, 0, stream>>>(prm);
    else
      decode_f32_kernel<128><<<blocks, 128, 0, stream>>>(prm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "decode (fp32): launch failed: %s", cudaGetErrorString(e));
    return PA_OK;
  }

  rc = get_encoder();
  if (rc != PA_OK) return rc;
  const int out_row_vecs = num_q_heads * head_dim * 2 / 16;
  plan_kernel<<<1, 1024, 0, stream>>>(prm, out_row_vecs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "decode: plan launch failed: %s", cudaGetErrorString(e));

  const DeviceState& st = g_dev[device];
  const int per_sm = st.ctas_per_sm[dtype == PA_BF16][head_dim == 128][group];
  const int grid = st.sms * (per_sm > 0 ? per_sm : 1);
  if (dtype == PA_BF16)
    return head_dim == 128 ? launch_tc<__nv_bfloat16, 128>(prm, k_cache, v_cache, dtype, stream, grid)
                           : launch_tc<__nv_bfloat16, 64>(prm, k_cache, v_cache, dtype, stream, grid);
  return head_dim == 128 ? launch_tc<__half, 128>(prm, k_cache, v_cache, dtype, stream, grid)
                         : launch_tc<__half, 64>(prm, k_cache, v_cache, dtype, stream, grid);
}

}  // extern "C"
