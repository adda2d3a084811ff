// kv_append and block_copy: the two bit-copy paths around decode attention,
// plus the per-device status word and pa_check_status.
//
// kv_append follows the OS-lab appendix "Lazy Allocation 与 Copy-on-Write 在
// LLM 推理系统中的应用", section 2.1 (each decode step appends the new
// token's K/V) with slots numbered physical * 16 + offset as in the
// "留书阁 / knowledge-20" block-table example.  block_copy follows the same
// appendix, section 4.4 (the writer gets a private copy of a shared block).
//
// Both are pure data movement in 16-byte vector loads/stores, consecutive
// threads on consecutive chunks so every warp moves whole 128-byte lines:
// kv_append one chunk per thread, the whole-block copies eight per thread.
// Both keep the default shared-memory / L1 split: their loads in flight need
// the L1 that the largest shared-memory split takes away (block copies ran
// 16-18 % slower with it, and a kernel that needs that split right after a
// small append started no later without it).
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "trace.h"
#include "pagedattn.h"
#include "status.h"

namespace pa {
namespace {

__device__ unsigned g_status_word;  // one per device; zero at module load

constexpr int kMaxDevices = 64;
constexpr int kMaxLayers = 256;
constexpr int kBlockSize = 16;

struct StatusSlot {
  std::once_flag once;
  unsigned* addr = nullptr;
};
StatusSlot g_slots[kMaxDevices];

// Token t's rows (heads_vecs 16-byte chunks: head h, chunk c of a row of
// 1 << row_shift) go to slot_mapping[t].  Threads (x, y) of a CTA: y picks a
// token, x walks its row, so no thread divides a flat index (the division
// by the row length, 64-bit, used to cost as much issue time as the copy).
__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                 const int64_t* __restrict__ slots, int num_tokens,
                                 int heads_vecs, int row_shift, int64_t num_slots,
                                 unsigned* status) {
  // Let the next kernel of the stream start its prologue now; touch memory only
  // once the kernel before this one has finished.
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();
  const int row_mask = (1 << row_shift) - 1;
  const int64_t num_heads = heads_vecs >> row_shift;
  for (int t = blockIdx.x * blockDim.y + threadIdx.y; t < num_tokens;
       t += gridDim.x * blockDim.y) {
    const int64_t slot = slots[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (threadIdx.x == 0) dev::flag_status(status, kStatusBounds);
      continue;
    }
    const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
    const uint4* kr = k + int64_t(t) * heads_vecs;
    const uint4* vr = v + int64_t(t) * heads_vecs;
    for (int j = threadIdx.x; j < heads_vecs; j += blockDim.x) {
      const int h = j >> row_shift, c = j & row_mask;
      const int64_t dst = (((blk * num_heads + h) * kBlockSize + off) << row_shift) + c;
      k_cache[dst] = kr[j];
      v_cache[dst] = vr[j];
    }
  }
}

struct LayerPtrs {
  uint4* k[kMaxLayers];
  uint4* v[kMaxLayers];
};

// One block's `block_vecs` 16-byte chunks, from -> to, by the whole CTA.
// Each thread issues eight loads before its eight stores, so an SM keeps
// enough bytes in flight to cover HBM (or CPU-GPU link) latency.  The two
// ranges must not overlap (a pair's source and destination are different
// blocks).
__device__ __forceinline__ void copy_block(const uint4* from, uint4* to, int block_vecs) {
  constexpr int kBatch = 8;
  for (int base = 0; base < block_vecs; base += kBatch * blockDim.x) {
    uint4 r[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      if (i < block_vecs) r[u] = from[i];
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      if (i < block_vecs) to[i] = r[u];
    }
  }
}

__global__ void block_copy_kernel(const __grid_constant__ LayerPtrs ptrs,
                                  const int64_t* __restrict__ pairs, int block_vecs,
                                  int64_t num_blocks, unsigned* status) {
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();
  const int pair = blockIdx.x, layer = blockIdx.y;
  const int64_t src = pairs[2 * int64_t(pair)], dst = pairs[2 * int64_t(pair) + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) dev::flag_status(status, kStatusBounds);
    return;
  }
  if (src == dst) return;
  uint4* base = blockIdx.z == 0 ? ptrs.k[layer] : ptrs.v[layer];
  copy_block(base + src * block_vecs, base + dst * block_vecs, block_vecs);
}

// Whole-block copies between two caches of the same shape (one on the
// device, one in page-locked host memory reached over the CPU-GPU link), all
// layers in one launch: grid (pair, layer, K/V).  Each thread keeps eight
// 16-byte loads in flight, so the link sees many outstanding requests.
__global__ void block_swap_kernel(const __grid_constant__ LayerPtrs src,
                                  const __grid_constant__ LayerPtrs dst,
                                  const int64_t* __restrict__ pairs, int block_vecs,
                                  int64_t num_src_blocks, int64_t num_dst_blocks,
                                  unsigned* status) {
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();
  const int pair = blockIdx.x, layer = blockIdx.y;
  const int64_t s = pairs[2 * int64_t(pair)], d = pairs[2 * int64_t(pair) + 1];
  if (s < 0 || s >= num_src_blocks || d < 0 || d >= num_dst_blocks) {
    if (threadIdx.x == 0) dev::flag_status(status, kStatusBounds);
    return;
  }
  const uint4* from = (blockIdx.z == 0 ? src.k[layer] : src.v[layer]) + s * block_vecs;
  uint4* to = (blockIdx.z == 0 ? dst.k[layer] : dst.v[layer]) + d * block_vecs;
  copy_block(from, to, block_vecs);
}

int elem_bytes(int dtype) { return dtype == PA_F32 ? 4 : 2; }

int check_common(int dtype, int head_dim, int num_kv_heads, int num_blocks, const char* who) {
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "%s: unknown dtype %d", who, dtype);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d (64 or 128)", who, head_dim);
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: num_kv_heads and num_blocks must be positive", who);
  return PA_OK;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

}  // namespace

unsigned* device_status_word() {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) {
    fail(PA_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  StatusSlot& slot = g_slots[device];
  std::call_once(slot.once, [&] {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) == cudaSuccess)
      slot.addr = static_cast<unsigned*>(addr);
  });
  if (!slot.addr) fail(PA_ERR_CUDA, "cudaGetSymbolAddress of the status word failed");
  return slot.addr;
}

}  // namespace pa

using namespace pa;

extern "C" {

PA_API int pa_kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                        int head_dim, int num_blocks, int dtype, void* stream) {
  PA_TRACE("pa_kv_append");
  int rc = check_common(dtype, head_dim, num_kv_heads, num_blocks, "kv_append");
  if (rc != PA_OK) return rc;
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "kv_append: num_tokens < 0");
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "kv_append: NULL pointer");
  if (misaligned(k) || misaligned(v) || misaligned(k_cache) || misaligned(v_cache))
    return fail(PA_ERR_INVALID_ARG, "kv_append: tensors must be 16-byte aligned");
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  const int row_vecs = head_dim * elem_bytes(dtype) / 16;  // 8, 16 or 32
  const int row_shift = row_vecs == 8 ? 3 : (row_vecs == 16 ? 4 : 5);
  const int heads_vecs = num_kv_heads * row_vecs;
  // 256 threads: x over a token's row, y over tokens
  const int tx = heads_vecs < 256 ? heads_vecs : 256, ty = 256 / tx;
  const int64_t want = (int64_t(num_tokens) + ty - 1) / ty;
  const int blocks = int(want < 65535 * 16 ? want : 65535 * 16);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(tx, ty);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<const uint4*>(k),
                                     static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
                                     static_cast<uint4*>(v_cache), slot_mapping, num_tokens,
                                     heads_vecs, row_shift, int64_t(num_blocks) * kBlockSize,
                                     status);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "kv_append: launch failed: %s", cudaGetErrorString(e));
  return PA_OK;
}

PA_API int pa_block_copy(void* const* k_caches, void* const* v_caches, int num_layers,
                         const int64_t* src_dst_pairs, int num_pairs, int num_kv_heads,
                         int head_dim, int num_blocks, int dtype, void* stream) {
  PA_TRACE("pa_block_copy");
  int rc = check_common(dtype, head_dim, num_kv_heads, num_blocks, "block_copy");
  if (rc != PA_OK) return rc;
  if (num_pairs < 0 || num_layers < 0 || num_layers > kMaxLayers)
    return fail(PA_ERR_INVALID_ARG, "block_copy: num_pairs < 0 or num_layers outside 0..%d",
                kMaxLayers);
  if (num_pairs == 0 || num_layers == 0) return PA_OK;
  if (!k_caches || !v_caches || !src_dst_pairs)
    return fail(PA_ERR_INVALID_ARG, "block_copy: NULL pointer");
  LayerPtrs ptrs = {};
  for (int l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || misaligned(k_caches[l]) || misaligned(v_caches[l]))
      return fail(PA_ERR_INVALID_ARG, "block_copy: layer %d cache pointer NULL or unaligned", l);
    ptrs.k[l] = static_cast<uint4*>(k_caches[l]);
    ptrs.v[l] = static_cast<uint4*>(v_caches[l]);
  }
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  const int block_vecs = num_kv_heads * kBlockSize * head_dim * elem_bytes(dtype) / 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_pairs, num_layers, 2);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, block_copy_kernel, ptrs, src_dst_pairs, block_vecs,
                                     int64_t(num_blocks), status);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "block_copy: launch failed: %s", cudaGetErrorString(e));
  return PA_OK;
}

PA_API int pa_block_swap(void* const* dev_k_caches, void* const* dev_v_caches,
                         void* const* host_k_caches, void* const* host_v_caches, int num_layers,
                         const int64_t* pairs, int num_pairs, int direction, int num_kv_heads,
                         int head_dim, int num_dev_blocks, int num_host_blocks, int dtype,
                         void* stream) {
  PA_TRACE("pa_block_swap");
  int rc = check_common(dtype, head_dim, num_kv_heads, num_dev_blocks, "block_swap");
  if (rc != PA_OK) return rc;
  if (num_host_blocks <= 0 || num_pairs < 0 || num_layers < 0 || num_layers > kMaxLayers ||
      (direction != PA_SWAP_OUT && direction != PA_SWAP_IN))
    return fail(PA_ERR_INVALID_ARG, "block_swap: bad num_host_blocks, num_pairs, num_layers or direction");
  if (num_pairs == 0 || num_layers == 0) return PA_OK;
  if (!dev_k_caches || !dev_v_caches || !host_k_caches || !host_v_caches || !pairs)
    return fail(PA_ERR_INVALID_ARG, "block_swap: NULL pointer");
  LayerPtrs dev = {}, host = {};
  for (int l = 0; l < num_layers; ++l) {
    void* hp[2] = {host_k_caches[l], host_v_caches[l]};
    void* dp[2] = {dev_k_caches[l], dev_v_caches[l]};
    for (int kv = 0; kv < 2; ++kv) {
      if (!dp[kv] || !hp[kv] || misaligned(dp[kv]) || misaligned(hp[kv]))
        return fail(PA_ERR_INVALID_ARG, "block_swap: layer %d pointer NULL or unaligned", l);
      // the host side must be page-locked memory the device can address
      cudaPointerAttributes a;
      if (cudaPointerGetAttributes(&a, hp[kv]) != cudaSuccess || a.type != cudaMemoryTypeHost ||
          !a.devicePointer) {
        cudaGetLastError();
        return fail(PA_ERR_INVALID_ARG, "block_swap: layer %d host cache is not page-locked host memory", l);
      }
      (kv ? host.v : host.k)[l] = static_cast<uint4*>(a.devicePointer);
      (kv ? dev.v : dev.k)[l] = static_cast<uint4*>(dp[kv]);
    }
  }
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  const int block_vecs = num_kv_heads * kBlockSize * head_dim * elem_bytes(dtype) / 16;
  const bool out = direction == PA_SWAP_OUT;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_pairs, num_layers, 2);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, block_swap_kernel, out ? dev : host, out ? host : dev,
                                     pairs, block_vecs,
                                     int64_t(out ? num_dev_blocks : num_host_blocks),
                                     int64_t(out ? num_host_blocks : num_dev_blocks), status);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "block_swap: launch failed: %s", cudaGetErrorString(e));
  return PA_OK;
}

PA_API int pa_check_status(void* stream) {
  unsigned* status = device_status_word();
  if (!status) return PA_ERR_CUDA;
  unsigned word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, status, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "check_status: %s", cudaGetErrorString(e));
  if (word & kStatusTimeout)
    return fail(PA_ERR_DEVICE_TIMEOUT, "a device-side wait ran out (status word 0x%x)", word);
  if (word & kStatusPlan)
    return fail(PA_ERR_INVALID_ARG,
                "a decode run found no plan for its shapes in the workspace (status 0x%x)", word);
  if (word & kStatusBounds)
    return fail(PA_ERR_DEVICE_BOUNDS, "a kernel saw an out-of-range block id, slot or length");
  return PA_OK;
}

}  // extern "C"
